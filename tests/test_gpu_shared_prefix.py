"""GPU parity of pa_decode_shared_prefix against the fp64 oracle.

Parallel samples of one prompt share the prompt's blocks (copy-on-write of
the last, partly filled or written-to block).  The shared-prefix decode
reads each group's shared blocks once for all of the group's query columns
(sample x head, in blocks of up to 64, the prefix in key chunks when it is
long), decodes every sample's own tokens separately and merges the partial
results.  Every case runs the whole step (copy_blocks, then the
decode with the new tokens appended) on NaN-poisoned pools and compares
with the oracle's step within the decode tolerance; the pools must come out
bit-identical to the oracle's.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, DevWorkload, host_bits, max_err

pytestmark = pytest.mark.gpu


def shared_prefix_len(w):
    """Tokens of the blocks every sample of a group names (the prompt's full
    blocks before the copied last one)."""
    pb = -(-w.meta["prompt_len"] // 16)
    return (pb - 1) * 16


def run(pa, w, append=True, prefix_len=None, group=None):
    dw = DevWorkload(w)
    pa.copy_blocks(dw.k, dw.v, dw.pairs)
    out = torch.full_like(dw.q, float("nan"))
    kw = dict(k_new=dw.k_new, v_new=dw.v_new, slot_mapping=dw.slots) if append else {}
    if not append:
        pa.reshape_and_cache(dw.k_new, dw.v_new, dw.k, dw.v, dw.slots)
    pa.decode_shared_prefix(out, dw.q, dw.k, dw.v, dw.tables, dw.lens,
                            group or w.meta["samples"],
                            shared_prefix_len(w) if prefix_len is None else prefix_len,
                            w.scale, **kw)
    torch.cuda.synchronize()
    return dw, out


@pytest.mark.parametrize("append", [True, False])
def test_parallel_sampling_config(pa, append):
    # 16 prompts x 8 samples, 40/8 heads (40 query columns per group and kv
    # head: five 8-column warps), 1024-token prompt: 1008 shared tokens
    w = synth.parsamp(poison=True)
    dw, out = run(pa, w, append)
    assert pa.get_device_error() == 0
    ref, k_ref, v_ref = oracle.step(w)
    assert max_err(out, ref) <= TOL[w.dtype]
    assert np.array_equal(host_bits(dw.k), k_ref) and np.array_equal(host_bits(dw.v), v_ref)


# A prompt that ends inside a block is copied from the original every step,
# so the samples' own tokens past the prompt in that block would not survive
# the copy (the NaN poison of the original's empty slots would reach the
# oracle): such prompts take no suffix here; block-aligned prompts do.
@pytest.mark.parametrize("prompts,samples,prompt_len,hq,hkv,d,dtype", [
    (2, 8, 40, 8, 2, 128, "f16"),      # unaligned prompt: 32 shared tokens, new token in the copy
    (3, 2, 304, 32, 8, 128, "bf16"),   # 8 columns: one consumer warp
    (2, 3, 512, 16, 1, 64, "f16"),     # 48 columns, group 16, head_dim 64
    (1, 16, 128, 8, 8, 64, "bf16"),    # MHA, 16 samples: 16 columns
    (4, 5, 1008, 12, 4, 128, "f16"),   # 15 columns
    (2, 4, 64, 64, 4, 128, "bf16"),    # group 16 x 4 samples = 64 columns
    (2, 4, 200, 16, 4, 64, "bf16"),    # unaligned, head_dim 64
    (1, 16, 2064, 16, 2, 128, "bf16"), # 128 columns (two column blocks), 2048 shared tokens in key chunks
    (2, 6, 1040, 24, 8, 64, "f16"),    # 18 columns (a half-used warp), head_dim 64, two key chunks
])
def test_shapes(pa, prompts, samples, prompt_len, hq, hkv, d, dtype):
    suffix = None if prompt_len % 16 == 0 else [0] * (prompts * samples)
    w = synth.parsamp(poison=True, num_prompts=prompts, samples=samples, prompt_len=prompt_len,
                      max_suffix=70, num_heads=hq, num_kv_heads=hkv, head_dim=d, dtype=dtype,
                      seed=prompts * 100 + samples, suffix_lens=suffix)
    dw, out = run(pa, w)
    assert pa.get_device_error() == 0
    ref, k_ref, v_ref = oracle.step(w)
    assert max_err(out, ref) <= TOL[w.dtype]
    assert np.array_equal(host_bits(dw.k), k_ref)


def test_shorter_shared_prefix_and_single_sample_groups(pa):
    # any multiple of 16 up to the shared blocks is a valid prefix, and a
    # group of one shares with nobody: both give the same result
    w = synth.parsamp(poison=True, num_prompts=4, samples=4, prompt_len=208, max_suffix=40,
                      num_heads=16, num_kv_heads=4, seed=9)
    ref, _, _ = oracle.step(w)
    for prefix_len, group in ((16, 4), (96, 4), (shared_prefix_len(w), 2), (64, 1)):
        _, out = run(pa, w, prefix_len=prefix_len, group=group)
        assert pa.get_device_error() == 0
        assert max_err(out, ref) <= TOL[w.dtype], (prefix_len, group)


def test_matches_plain_decode(pa):
    w = synth.parsamp(poison=True, num_prompts=4, samples=8, prompt_len=512, max_suffix=100,
                      seed=31)
    dw, out = run(pa, w)
    b = DevWorkload(w)
    pa.copy_blocks(b.k, b.v, b.pairs)
    pa.decode_append(b.out, b.q, b.k, b.v, b.tables, b.lens, b.k_new, b.v_new, b.slots, w.scale)
    torch.cuda.synchronize()
    assert float((out.float() - b.out.float()).abs().max()) <= TOL[w.dtype]
    assert torch.equal(dw.k.view(torch.int16), b.k.view(torch.int16))


def test_bad_arguments(pa):
    w = synth.parsamp(num_prompts=2, samples=4, prompt_len=64, max_suffix=10)
    dw = DevWorkload(w)
    for group, prefix in ((3, 48), (4, 40), (4, 0), (0, 48)):
        with pytest.raises(pa.PagedAttnError) as e:
            pa.decode_shared_prefix(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, group, prefix,
                                    w.scale)
        assert e.value.status in (1, 3)


def test_sequence_shorter_than_prefix_is_flagged(pa):
    w = synth.parsamp(num_prompts=2, samples=4, prompt_len=64, max_suffix=10)
    dw = DevWorkload(w)
    dw.lens[1] = 20
    pa.decode_shared_prefix(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, 4, 48, w.scale)
    assert pa.get_device_error() & pa.DEVERR["SEQLEN_RANGE"]


def test_bad_prefix_table_entry_is_reported(pa):
    # a prefix entry past the pool: the prefix kernel reads a valid block in
    # its place and records the table error
    w = synth.parsamp(num_prompts=2, samples=4, prompt_len=512, max_suffix=10, seed=13)
    dw = DevWorkload(w)
    dw.tables[0, 3] = w.k_cache.shape[0] + 5          # group 0's first table names the prefix
    pa.get_device_error()
    pa.decode_shared_prefix(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, 4, 496, w.scale)
    torch.cuda.synchronize()
    assert pa.get_device_error() & pa.DEVERR["TABLE_RANGE"]


def test_repeated_calls_give_the_same_bits(pa):
    # the prefix chunks, the suffix split and the merge order are fixed by
    # the shapes alone, so a repeated call reproduces the output bit for bit
    w = synth.parsamp(num_prompts=4, samples=8, prompt_len=2048, max_suffix=100, seed=17)
    dw = DevWorkload(w)
    pa.copy_blocks(dw.k, dw.v, dw.pairs)
    pa.reshape_and_cache(dw.k_new, dw.v_new, dw.k, dw.v, dw.slots)
    outs = []
    for _ in range(2):
        out = torch.full_like(dw.q, float("nan"))
        pa.decode_shared_prefix(out, dw.q, dw.k, dw.v, dw.tables, dw.lens, 8,
                                shared_prefix_len(w), w.scale)
        torch.cuda.synchronize()
        outs.append(out)
    assert pa.get_device_error() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    ref, _, _ = oracle.step(w)
    assert max_err(outs[1], ref) <= TOL[w.dtype]


@pytest.mark.parametrize("prompt_len,hq,hkv,suffix", [
    (64, 8, 2, [3000, 5000]),     # suffix runs cut into far more than 32 pieces
    (16384, 4, 1, [700, 1500]),   # and a prefix in more than 32 key chunks
])
def test_long_suffixes_cut_into_many_pieces(pa, prompt_len, hq, hkv, suffix):
    # the suffix decode's balanced split cuts each long suffix run into many
    # pieces, which the final merge folds together with the prefix chunks
    w = synth.parsamp(poison=True, num_prompts=1, samples=2, prompt_len=prompt_len,
                      num_heads=hq, num_kv_heads=hkv, head_dim=128, dtype="bf16", seed=23,
                      suffix_lens=suffix)
    dw, out = run(pa, w)
    assert pa.get_device_error() == 0
    ref, k_ref, v_ref = oracle.step(w)
    assert max_err(out, ref) <= TOL[w.dtype]
    assert np.array_equal(host_bits(dw.k), k_ref) and np.array_equal(host_bits(dw.v), v_ref)


def test_workspace_reused_between_split_and_whole_suffix_decodes(pa):
    # One workspace, filled with 0xff bytes before every call, serves a batch
    # whose suffix runs the balanced split cuts (wide tables), then one whose
    # tables are narrow enough to be decoded a run a warp, then the first
    # again: the record of which runs were cut must never leak from a call
    # into the next.
    wa = synth.parsamp(poison=True, num_prompts=2, samples=4, prompt_len=512, max_suffix=200,
                       num_heads=8, num_kv_heads=2, seed=41)
    wb = synth.parsamp(poison=True, num_prompts=2, samples=4, prompt_len=48, max_suffix=40,
                       num_heads=8, num_kv_heads=2, seed=42)
    assert wa.block_tables.shape[1] > 8 >= wb.block_tables.shape[1]
    need = max(pa.decode_shared_prefix_workspace_size(w.num_seqs, w.meta["samples"],
                                                      shared_prefix_len(w), w.num_heads,
                                                      w.num_kv_heads, w.head_dim,
                                                      w.block_tables.shape[1]) for w in (wa, wb))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for w in (wa, wb, wa):
        dw = DevWorkload(w)
        pa.copy_blocks(dw.k, dw.v, dw.pairs)
        ws.fill_(0xff)
        out = torch.full_like(dw.q, float("nan"))
        pa.decode_shared_prefix(out, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.meta["samples"],
                                shared_prefix_len(w), w.scale, k_new=dw.k_new, v_new=dw.v_new,
                                slot_mapping=dw.slots, workspace=ws)
        torch.cuda.synchronize()
        assert pa.get_device_error() == 0
        ref, _, _ = oracle.step(w)
        assert max_err(out, ref) <= TOL[w.dtype]
