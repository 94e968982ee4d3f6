"""GPU parity of the pool kernels: reshape_and_cache, copy_blocks, gather_kv
and validate_tables, bit-exact against the oracle (whole pools compared as raw
16-bit patterns, so slots that must not change are checked too)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import DevWorkload, dev_bits, host_bits

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_page3_figure_gather(pa):
    g = json.load(open(os.path.join(GOLDEN, "page3_block_table.json")))
    nb, hkv, d = g["pool_blocks"], 2, 64
    tag = (np.arange(nb)[:, None] * 16 + np.arange(16)[None, :]).astype(np.float16)
    pool = np.broadcast_to(tag[:, None, :, None], (nb, hkv, 16, d)).copy().view(np.uint16)
    k = dev_bits(pool, "f16")
    v = dev_bits(pool, "f16")
    tables = torch.tensor([g["tables"]["A"], g["tables"]["B"]], dtype=torch.int32, device="cuda")
    lens = torch.tensor([48, 40], dtype=torch.int32, device="cuda")
    ko = torch.zeros(2, hkv, 48, d, dtype=torch.float16, device="cuda")
    vo = torch.zeros_like(ko)
    pa.gather_kv(ko, vo, k, v, tables, lens)
    got = ko[:, 0, :, 0].float().cpu().numpy()
    for s, (req, L) in enumerate([("A", 48), ("B", 40)]):
        want = [b * 16 + o for b in g["tables"][req] for o in range(16)][:L]
        assert got[s, :L].astype(int).tolist() == want
    assert torch.equal(ko, vo)
    assert pa.get_device_error() == 0


@pytest.mark.parametrize("name", ["tiny", "gqa8b"])
def test_gather_matches_oracle(pa, name):
    w = synth.by_name(name, poison=True) if name == "tiny" else synth.gqa8b(num_seqs=16, poison=True)
    dw = DevWorkload(w)
    mb = w.max_blocks_per_seq
    ko = torch.zeros(w.num_seqs, w.num_kv_heads, mb * 16, w.head_dim, dtype=dw.k.dtype, device="cuda")
    vo = torch.zeros_like(ko)
    pa.gather_kv(ko, vo, dw.k, dw.v, dw.tables, dw.lens)
    kh, vh = host_bits(ko), host_bits(vo)
    for s, L in enumerate(w.seq_lens):
        rk, rv = oracle.gather_kv(w.k_cache, w.v_cache, w.block_tables, s, int(L))
        assert np.array_equal(kh[s, :, :L], rk) and np.array_equal(vh[s, :, :L], rv)
    assert pa.get_device_error() == 0


@pytest.mark.parametrize("name", ["tiny", "gqa8b", "parsamp_small"])
def test_reshape_and_cache_bit_exact(pa, name):
    if name == "parsamp_small":
        w = synth.parsamp(num_prompts=2, samples=4, prompt_len=40, suffix_lens=[0] * 8,
                          num_heads=8, num_kv_heads=2, head_dim=64, poison=True)
    elif name == "tiny":
        w = synth.tiny(poison=True)
    else:
        w = synth.gqa8b(poison=True)
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[1] = -1                          # a padding token
    dw = DevWorkload(w)
    pa.reshape_and_cache(dw.k_new, dw.v_new, dw.k, dw.v, dw.slots)
    k, v = w.k_cache.copy(), w.v_cache.copy()
    oracle.reshape_and_cache(k, v, w.k_new, w.v_new, w.slot_mapping)
    assert np.array_equal(host_bits(dw.k), k)
    assert np.array_equal(host_bits(dw.v), v)
    assert pa.get_device_error() == 0


def test_reshape_and_cache_slot_past_pool(pa):
    w = synth.tiny()
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[2] = w.num_blocks * 16 + 5
    dw = DevWorkload(w)
    pa.reshape_and_cache(dw.k_new, dw.v_new, dw.k, dw.v, dw.slots)
    k, v = w.k_cache.copy(), w.v_cache.copy()
    assert oracle.reshape_and_cache(k, v, w.k_new, w.v_new, w.slot_mapping) == 1
    assert np.array_equal(host_bits(dw.k), k) and np.array_equal(host_bits(dw.v), v)
    assert pa.get_device_error() == pa.DEVERR["SLOT_RANGE"]


@pytest.mark.parametrize("D,hkv,layout", [(128, 4, "blocks"), (64, 3, "scatter")])
def test_reshape_and_cache_many_tokens(pa, D, hkv, layout):
    # a prefill-sized write: several grid strides of the kernel and a ragged
    # tail, with padding tokens; whole blocks in order or random distinct slots
    rng = np.random.default_rng(77 + D)
    nb, ntok = 2600, 20011
    if layout == "blocks":
        blocks = rng.choice(nb, -(-ntok // 16), replace=False)
        slots = (blocks[:, None] * 16 + np.arange(16)[None, :]).reshape(-1)[:ntok]
    else:
        slots = rng.choice(nb * 16, ntok, replace=False)
    slots = slots.astype(np.int64)
    slots[rng.choice(ntok, 37, replace=False)] = -1
    k = rng.integers(0, 1 << 16, (nb, hkv, 16, D), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, (nb, hkv, 16, D), dtype=np.uint16)
    kn = rng.integers(0, 1 << 16, (ntok, hkv, D), dtype=np.uint16)
    vn = rng.integers(0, 1 << 16, (ntok, hkv, D), dtype=np.uint16)
    dk, dv = dev_bits(k, "bf16"), dev_bits(v, "bf16")
    pa.reshape_and_cache(dev_bits(kn, "bf16"), dev_bits(vn, "bf16"), dk, dv,
                         torch.from_numpy(slots).cuda())
    assert oracle.reshape_and_cache(k, v, kn, vn, slots) == 0
    assert np.array_equal(host_bits(dk), k) and np.array_equal(host_bits(dv), v)
    assert pa.get_device_error() == 0


@pytest.mark.parametrize("D", [64, 128])
def test_copy_blocks_bit_exact(pa, D):
    w = synth.parsamp(num_prompts=3, samples=5, prompt_len=72, max_suffix=30, num_heads=8,
                      num_kv_heads=4, head_dim=D, dtype="bf16", poison=True)
    dw = DevWorkload(w)
    pa.copy_blocks(dw.k, dw.v, dw.pairs)
    k, v = w.k_cache.copy(), w.v_cache.copy()
    assert oracle.copy_blocks(k, v, w.block_mapping) == 0
    assert np.array_equal(host_bits(dw.k), k) and np.array_equal(host_bits(dw.v), v)
    assert pa.get_device_error() == 0


def test_copy_blocks_bad_pair_is_skipped(pa):
    w = synth.parsamp(num_prompts=1, samples=3, prompt_len=32, max_suffix=8, num_heads=4,
                      num_kv_heads=2, head_dim=64)
    pairs = np.concatenate([w.block_mapping, [[0, w.num_blocks + 3]]]).astype(np.int64)
    dw = DevWorkload(w)
    pa.copy_blocks(dw.k, dw.v, torch.from_numpy(pairs).cuda())
    k, v = w.k_cache.copy(), w.v_cache.copy()
    assert oracle.copy_blocks(k, v, pairs) == 1
    assert np.array_equal(host_bits(dw.k), k) and np.array_equal(host_bits(dw.v), v)
    assert pa.get_device_error() == pa.DEVERR["BLOCK_RANGE"]


def test_copy_blocks_many_pairs(pa):
    # more pairs than one launch's grid.y allows
    nb, hkv, d = 70000, 1, 64
    k = torch.randn(nb, hkv, 16, d, device="cuda").half()
    v = torch.randn_like(k)
    src = torch.arange(0, 33000, device="cuda", dtype=torch.int64)
    dst = src + 35000
    pairs = torch.stack([src, dst], 1).contiguous()
    k0, v0 = k.clone(), v.clone()
    pa.copy_blocks(k, v, pairs)
    assert torch.equal(k[35000:68000], k0[:33000]) and torch.equal(v[35000:68000], v0[:33000])
    assert torch.equal(k[:35000], k0[:35000]) and torch.equal(k[68000:], k0[68000:])


def test_validate_tables_counts_bad_entries(pa):
    w = synth.tiny()
    tables = w.block_tables.copy()
    tables[0, 0] = w.num_blocks          # read by the decode: bad
    tables[1, -1] = 9999                 # past the sequence's blocks: never read
    lens = w.seq_lens.copy()
    lens[2] = -3                         # bad length
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.validate_tables(torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                       w.num_blocks, cnt)
    n_read_bad = int(tables[1, -1] == 9999 and (w.seq_lens[1] + 15) // 16 == tables.shape[1])
    assert int(cnt.item()) == 2 + n_read_bad


def test_bounded_wait_gives_up_and_reports(pa):
    # a copy wait that nothing completes: the kernel must time out, flag it,
    # finish, and leave the context usable
    assert pa.get_device_error() == 0
    pa.selftest_bounded_wait(2000)
    assert pa.get_device_error() == pa.DEVERR["TIMEOUT"]
    w = synth.tiny(poison=True)
    dw = DevWorkload(w)
    dw.step(pa)
    ref, _, _ = oracle.step(w)
    assert float(np.abs(dw.out.float().cpu().numpy() - ref).max()) <= 4e-3
    assert pa.get_device_error() == 0
