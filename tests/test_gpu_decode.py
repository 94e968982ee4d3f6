"""GPU parity of paged decode attention against the fp64 oracle.

Every case runs the whole decode step through the C ABI on seeded inputs in
which slots holding no live token are NaN (so any over-read or wrong-table
read shows), and compares element by element within the stated tolerance:
max |err| <= 4e-3 for fp16 outputs, 1.6e-2 for bf16.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, DevWorkload, dev_bits, host_bits, max_err, to_f64

pytestmark = pytest.mark.gpu

MODES = [-1, 0, 16, 64, 512]          # no split, balanced split, fixed partitions


def check(pa, w, partition_size=0, ws=None):
    dw = DevWorkload(w)
    dw.step(pa, partition_size=partition_size, workspace=ws)
    ref, k_ref, v_ref = oracle.step(w)
    err = max_err(dw.out, ref)
    assert err <= TOL[w.dtype], f"max|err| {err}"
    assert pa.get_device_error() == 0
    return dw, ref


LENS = [0, 1, 2, 15, 16, 17, 31, 33, 100, 257, 700, 1029]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("Hq,Hkv,D,dtype", [
    (8, 8, 64, "f16"), (8, 8, 128, "bf16"), (8, 4, 128, "f16"), (12, 4, 64, "bf16"),
    (16, 4, 128, "bf16"), (10, 2, 128, "f16"), (12, 2, 64, "f16"), (14, 2, 128, "bf16"),
    (16, 2, 128, "f16"), (8, 1, 64, "bf16"),
    # groups 9..16: the query columns take a second 8-column tile (MQA-like
    # sharing of one kv head by many query heads)
    (9, 1, 128, "f16"), (26, 2, 128, "bf16"), (15, 1, 64, "bf16"), (16, 1, 128, "bf16"),
    (32, 2, 64, "f16")])
def test_decode_ragged(pa, mode, Hq, Hkv, D, dtype):
    w = synth.build("ragged", len(LENS), Hq, Hkv, D, dtype, LENS, seed=100 + Hq + D, append=True,
                    poison=True)
    check(pa, w, mode)


@pytest.mark.parametrize("name", ["tiny", "mha7b", "gqa8b", "parsamp"])
def test_configs_reduced(pa, name):
    if name == "tiny":
        w = synth.tiny(poison=True)
    elif name == "mha7b":
        w = synth.mha7b(poison=True, num_seqs=8)
    elif name == "gqa8b":
        w = synth.gqa8b(poison=True, num_seqs=32)
    else:
        w = synth.parsamp(poison=True, num_prompts=2, samples=8)
    for mode in (0, -1, 512):
        check(pa, w, mode)


def test_long_reduced_split_k(pa):
    w = synth.long(poison=True, lens=(4096, 8192, 12288 + 5, 16384 - 7))
    check(pa, w, 512)
    check(pa, w, 0)


def test_seq_len_one_returns_v_exactly(pa):
    w = synth.build("one", 6, 16, 4, 128, "bf16", [1] * 6, seed=3)
    dw = DevWorkload(w)
    pa.decode(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale)
    out = host_bits(dw.out)
    for s in range(6):
        for h in range(16):
            assert np.array_equal(out[s, h], w.v_cache[w.block_tables[s, 0], h // 4, 0])


def test_identical_keys_give_mean_of_v(pa):
    w = synth.build("same", 4, 8, 2, 128, "f16", [5, 40, 333, 1000], seed=4)
    w.k_cache = w.k_cache.copy()
    w.k_cache[:] = w.k_cache[0, :, 0:1, :]
    dw = DevWorkload(w)
    pa.decode(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale)
    got = to_f64(dw.out)
    for s, L in enumerate(w.seq_lens):
        _, vv = oracle.gather_kv(w.k_cache, w.v_cache, w.block_tables, s, int(L))
        mean = oracle.decode_bits(vv, "f16").mean(axis=1)
        for h in range(8):
            assert np.abs(got[s, h] - mean[h // 4]).max() <= TOL["f16"]


def test_block_permutation_is_bit_exact(pa):
    w = synth.build("perm", 5, 16, 4, 128, "bf16", [3, 64, 300, 999, 17], seed=8, pool_factor=2.0)
    dw = DevWorkload(w)
    pa.decode(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale)
    base = dw.out.clone()
    perm = np.random.default_rng(1).permutation(w.num_blocks)
    k2 = np.empty_like(w.k_cache)
    v2 = np.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    t2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    out2 = torch.empty_like(dw.q)
    pa.decode(out2, dw.q, dev_bits(k2, "bf16"), dev_bits(v2, "bf16"),
              torch.from_numpy(t2).cuda(), dw.lens, w.scale)
    assert torch.equal(out2, base)


def test_cow_remap_is_bit_exact(pa):
    w = synth.parsamp(num_prompts=2, samples=8, prompt_len=64, max_suffix=40)
    dw = DevWorkload(w)
    pa.reshape_and_cache(dw.k_new, dw.v_new, dw.k, dw.v, dw.slots)
    before = torch.empty_like(dw.q)
    pa.decode(before, dw.q, dw.k, dw.v, torch.from_numpy(w.tables_before_cow).cuda(), dw.lens,
              w.scale)
    pa.copy_blocks(dw.k, dw.v, dw.pairs)
    pa.decode(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale)
    assert torch.equal(before, dw.out)


def test_cow_unaligned_prefix_no_crosstalk(pa):
    kw = dict(num_prompts=2, samples=4, prompt_len=40, suffix_lens=[0] * 8, num_heads=8,
              num_kv_heads=2, head_dim=128, poison=True)
    w = synth.parsamp(**kw)
    dw, ref = check(pa, w, 0)
    w2 = synth.parsamp(**kw)
    w2.k_new = w2.k_new.copy()
    w2.k_new[5] = synth.to_bits(np.full(w2.k_new[5].shape, 2.0, np.float32), "f16")
    dw2, ref2 = check(pa, w2, 0)
    diff = (dw.out != dw2.out).flatten(1).any(1).cpu().numpy()
    assert diff.tolist() == [s == 5 for s in range(8)]


def test_fixed_partials_match_oracle(pa):
    P = 64
    w = synth.build("parts", 5, 16, 4, 128, "f16", [17, 64, 65, 300, 1000], seed=12, poison=True)
    dw = DevWorkload(w)
    ws = pa.workspace_for(dw.q, dw.k, dw.tables, P)
    pa.decode(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale, partition_size=P,
              workspace=ws)
    torch.cuda.synchronize()
    S, Hq, D = w.q.shape
    pmax = -(-w.max_blocks_per_seq * 16 // P)
    rows = S * Hq * pmax

    def up(x):
        return (x + 255) // 256 * 256

    raw = ws.cpu().numpy()
    l_off = up(4 * rows)
    o_off = up(l_off + 4 * rows)
    gm = raw[:4 * rows].view(np.float32).reshape(S, Hq, pmax)
    gl = raw[l_off:l_off + 4 * rows].view(np.float32).reshape(S, Hq, pmax)
    go = raw[o_off:o_off + 4 * rows * D].view(np.float32).reshape(S, Hq, pmax, D)
    m, l, o = oracle.partials(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale,
                              "f16", P, max_partitions=pmax)
    for s, L in enumerate(w.seq_lens):
        n = -(-int(L) // P)
        if n <= 1:
            continue                      # a single partition is written as the output itself
        np.testing.assert_allclose(gm[s, :, :n], m[s, :, :n], rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(gl[s, :, :n], l[s, :, :n], rtol=1e-4, atol=1e-5)
        # the weights enter the second product rounded to fp16 (relative error
        # <= 2^-11), so a normalised partial output moves by <= 2^-11 max|v|
        _, vv = oracle.gather_kv(w.k_cache, w.v_cache, w.block_tables, s, int(L))
        vmax = float(np.abs(oracle.decode_bits(vv, "f16")).max())
        np.testing.assert_allclose(go[s, :, :n], o[s, :, :n], rtol=0, atol=2.0 ** -11 * vmax + 1e-5)


def test_single_partition_equals_no_split(pa):
    # with partitions longer than every sequence the split only cuts runs to
    # balance the warps; the merge is exact in real arithmetic, so the result
    # agrees with the unsplit decode up to rounding
    w = synth.build("one_part", 6, 32, 8, 128, "bf16", [5, 16, 100, 511, 512, 300], seed=13)
    dw = DevWorkload(w)
    pa.decode(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale, partition_size=-1)
    a = dw.out.clone()
    pa.decode(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale, partition_size=512)
    assert float((a.float() - dw.out.float()).abs().max()) <= TOL["bf16"]


def test_repeatable(pa):
    w = synth.gqa8b(num_seqs=24)
    dw = DevWorkload(w)
    pa.decode(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale)
    a = dw.out.clone()
    pa.decode(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale)
    assert torch.equal(a, dw.out)


def test_all_empty_and_zero_scale(pa):
    w = synth.build("empty", 3, 8, 2, 64, "f16", [0, 0, 0], seed=1, pool_blocks=4, max_blocks=2)
    dw = DevWorkload(w)
    dw.out.fill_(1.0)
    pa.decode(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale)
    assert torch.count_nonzero(dw.out) == 0
    w = synth.build("scale0", 3, 8, 2, 64, "f16", [7, 70, 700], seed=2, scale=0.0)
    check(pa, w, 0)


def test_many_short_sequences(pa):
    rng = np.random.default_rng(5)
    lens = rng.integers(0, 40, size=3000)
    w = synth.build("many", 3000, 8, 1, 64, "bf16", lens, seed=6, poison=True)
    check(pa, w, 0)
    check(pa, w, -1)


@pytest.mark.parametrize("n", [1, 7, 100, 2047, 2048, 2049, 5000])
def test_batch_sizes_across_kernel_variants(pa, n):
    # Up to 2048 sequences each decode block keeps the per-sequence lengths
    # and unit prefix in its shared memory; larger batches have a one-block
    # kernel build them once in the workspace.  Batch sizes on both sides of
    # that edge match the oracle.
    rng = np.random.default_rng(n)
    lens = rng.integers(0, 48, size=n)
    w = synth.build("sizes", n, 16, 4, 128, "bf16", lens, seed=n, poison=True)
    check(pa, w, 0)


@pytest.mark.parametrize("mode", [0, -1, 64])
@pytest.mark.parametrize("Hq,Hkv,D,dtype", [(16, 1, 64, "f16"), (8, 2, 128, "bf16")])
def test_twenty_thousand_ragged_sequences(pa, mode, Hq, Hkv, D, dtype):
    # a continuous batch far above the shared-memory edge, at group 16 and 4,
    # lengths 0..300 with NaN in every slot no live token holds
    n = 20000
    rng = np.random.default_rng(2000 + Hq)
    lens = rng.integers(0, 301, size=n)
    lens[rng.integers(0, n, size=50)] = 0
    w = synth.build("b20k", n, Hq, Hkv, D, dtype, lens, seed=2001 + Hq, append=True, poison=True)
    check(pa, w, mode)


def test_group_above_sixteen_is_refused(pa):
    w = synth.build("g17", 2, 17, 1, 64, "f16", [5, 9], seed=3)
    dw = DevWorkload(w)
    with pytest.raises(pa.PagedAttnError) as e:
        pa.decode(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale)
    assert e.value.status == 2                         # PA_ERR_UNSUPPORTED


def test_bad_table_entry_is_flagged_not_faulting(pa):
    w = synth.build("badtab", 3, 8, 2, 64, "f16", [20, 40, 60], seed=9)
    w.block_tables = w.block_tables.copy()
    w.block_tables[1, 1] = w.num_blocks + 100
    dw = DevWorkload(w)
    pa.decode(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale)
    assert pa.get_device_error() & pa.DEVERR["TABLE_RANGE"]


def test_bad_seq_len_is_flagged(pa):
    w = synth.build("badlen", 3, 8, 2, 64, "f16", [20, 40, 60], seed=9)
    dw = DevWorkload(w)
    dw.lens[1] = 10 ** 6
    pa.decode(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale)
    assert pa.get_device_error() & pa.DEVERR["SEQLEN_RANGE"]


def test_workspace_too_small(pa):
    w = synth.build("ws", 3, 8, 2, 64, "f16", [20, 400, 60], seed=9)
    dw = DevWorkload(w)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PagedAttnError) as e:
        pa.decode(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale, partition_size=64,
                  workspace=small)
    assert e.value.status == 3


def test_other_stream(pa):
    w = synth.gqa8b(num_seqs=8, poison=True)
    dw = DevWorkload(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dw.step(pa)
    s.synchronize()
    ref, _, _ = oracle.step(w)
    assert max_err(dw.out, ref) <= TOL["bf16"]


def test_balanced_workspace_reused_across_shapes(pa):
    # The workspace's contents need no initialisation: one buffer, filled with
    # 0xff bytes (NaN as fp32, -1 as descriptors) before every call, serves
    # calls of several shapes in turn -- groups 4, 7 and 8, head_dim 64 and
    # 128, runs cut into one to dozens of pieces -- and every result stays
    # within tolerance, twice over.
    rng = np.random.default_rng(74)
    cases = [
        synth.build("reuse_a", 6, 32, 8, 128, "bf16", [5, 900, 3000, 17, 1200, 64], seed=71,
                    append=True, poison=True),
        synth.build("reuse_b", 5, 14, 2, 64, "f16", [4000, 33, 2500, 1, 700], seed=72,
                    poison=True),
        synth.long(poison=True, lens=(8192, 16384 + 3), partition_size=0),
        synth.build("reuse_d", 40, 16, 2, 128, "f16", rng.integers(0, 2000, size=40), seed=73,
                    poison=True),
    ]
    need = max(pa.decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                        w.block_tables.shape[1], 0) for w in cases)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        for w in cases:
            ws.fill_(0xFF)
            check(pa, w, 0, ws=ws)


@pytest.mark.parametrize("append", [False, True])
@pytest.mark.parametrize("mode", [0, 512])
def test_back_to_back_steps_in_a_cuda_graph(pa, mode, append):
    # The configuration the bench times: decode calls captured back to back
    # in one CUDA graph, each a programmatic dependent launch of the call
    # before, sharing one output buffer, one pool and one workspace.  Every
    # step has its own queries and lengths (and, with append, its own new
    # token written into the pool on the way), so the runs are cut in
    # different places from step to step.  After each replay the output is
    # the last step's over the pool all the steps left, and it matches the
    # oracle.  A step that overtook the previous step's merge would leave
    # that merge's rows, or read its slots, in the result.
    rng = np.random.default_rng(91 + mode + append)
    base = np.clip(np.round(rng.lognormal(np.log(600), 1.0, size=48)), 16, 4096).astype(int)
    w = synth.build("b2b", 48, 32, 8, 128, "bf16", base, seed=92 + mode, poison=True)
    dw = DevWorkload(w)
    steps = 5
    qs, lens, news = [], [], []
    k_host, v_host = w.k_cache.copy(), w.v_cache.copy()
    for i in range(steps):
        q = synth.to_bits(rng.standard_normal(w.q.shape).astype(np.float32), w.dtype)
        L = np.minimum(w.seq_lens, rng.integers(1, 4097, size=w.num_seqs)).astype(np.int32)
        if i == steps - 1:
            L[::7] = w.seq_lens[::7]
        qs.append(q)
        lens.append(L)
        if append:
            shape = (w.num_seqs, w.num_kv_heads, w.head_dim)
            kn = synth.to_bits(rng.standard_normal(shape).astype(np.float32), w.dtype)
            vn = synth.to_bits(rng.standard_normal(shape).astype(np.float32), w.dtype)
            pos = L - 1
            slots = (w.block_tables[np.arange(w.num_seqs), pos // 16].astype(np.int64) * 16
                     + pos % 16)
            oracle.reshape_and_cache(k_host, v_host, kn, vn, slots)
            news.append((dev_bits(kn, w.dtype), dev_bits(vn, w.dtype),
                         torch.from_numpy(slots).cuda()))
    q_dev = [dev_bits(q, w.dtype) for q in qs]
    l_dev = [torch.from_numpy(L).cuda() for L in lens]
    ws = pa.workspace_for(dw.q, dw.k, dw.tables, mode)

    def step(i, stream):
        if append:
            kn, vn, sl = news[i]
            pa.decode_append(dw.out, q_dev[i], dw.k, dw.v, dw.tables, l_dev[i], kn, vn, sl,
                             w.scale, partition_size=mode, workspace=ws, stream=stream)
        else:
            pa.decode(dw.out, q_dev[i], dw.k, dw.v, dw.tables, l_dev[i], w.scale,
                      partition_size=mode, workspace=ws, stream=stream)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(steps):                                     # warm-up
            step(i, s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(steps):
                step(i, s)
    torch.cuda.current_stream().wait_stream(s)
    ref = oracle.decode(qs[-1], k_host, v_host, w.block_tables, lens[-1], w.scale, w.dtype)
    for _ in range(3):
        dw.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert max_err(dw.out, ref) <= TOL[w.dtype]
    assert pa.get_device_error() == 0
    if append:
        assert np.array_equal(host_bits(dw.k), k_host) and np.array_equal(host_bits(dw.v), v_host)


# ---------------------------------------------------------------------------
# pa_decode_append: reshape_and_cache + decode in one launch
# ---------------------------------------------------------------------------
def _append_cases():
    return {
        "tiny": synth.tiny(poison=True),
        "gqa8b": synth.gqa8b(num_seqs=24, poison=True),
        "ragged": synth.build("ragged", len(LENS), 16, 4, 128, "bf16", LENS, seed=55, append=True,
                              poison=True),
        "parsamp": synth.parsamp(num_prompts=2, samples=4, prompt_len=40, suffix_lens=[0] * 8,
                                 num_heads=8, num_kv_heads=2, head_dim=64, poison=True),
    }


@pytest.mark.parametrize("mode", [-1, 0, 64])
@pytest.mark.parametrize("name", ["tiny", "gqa8b", "ragged", "parsamp"])
def test_decode_append_equals_separate_steps(pa, name, mode):
    w = _append_cases()[name]
    a = DevWorkload(w)
    a.step(pa, partition_size=mode)                      # copy, reshape, decode
    b = DevWorkload(w)
    if b.pairs is not None:
        pa.copy_blocks(b.k, b.v, b.pairs)
    pa.decode_append(b.out, b.q, b.k, b.v, b.tables, b.lens, b.k_new, b.v_new, b.slots, w.scale,
                     partition_size=mode)
    assert torch.equal(a.out, b.out)
    # pools hold NaN in unused slots: compare raw 16-bit patterns
    assert torch.equal(a.k.view(torch.int16), b.k.view(torch.int16))
    assert torch.equal(a.v.view(torch.int16), b.v.view(torch.int16))
    assert pa.get_device_error() == 0
    ref, k_ref, v_ref = oracle.step(w)
    assert max_err(b.out, ref) <= TOL[w.dtype]
    assert np.array_equal(host_bits(b.k), k_ref) and np.array_equal(host_bits(b.v), v_ref)


def test_decode_append_rejects_a_slot_not_at_the_end(pa):
    w = synth.tiny()
    dw = DevWorkload(w)
    k0 = dw.k.clone()
    slots = dw.slots.clone()
    s = int(np.argmax(w.seq_lens))                       # a sequence with several tokens
    L = int(w.seq_lens[s])
    pos = L - 2                                          # not the newest position
    slots[s] = int(w.block_tables[s, pos // 16]) * 16 + pos % 16
    pa.decode_append(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, dw.k_new, dw.v_new, slots,
                     w.scale)
    assert pa.get_device_error() & pa.DEVERR["APPEND_SLOT"]
    blk, off = slots[s].item() // 16, slots[s].item() % 16
    assert torch.equal(dw.k[blk, :, off], k0[blk, :, off])   # that token was not written
