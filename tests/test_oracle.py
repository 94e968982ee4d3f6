"""Pins of the fp64 oracle against what the pages and mathematics fix.

CPU only.  Each test ties the oracle to something other than itself: the
block-table figure of the vLLM reading notes, the KV-size worked example of
the mlsys course page, a library routine (torch's fp64 scaled-dot-product
attention, numpy's / torch's 16-bit decoders), closed forms of softmax
attention, invariances the method must have, and a pure-Python brute force.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import brute
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f16_bits(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def small(num_seqs=3, Hq=4, Hkv=2, D=16, dtype="f16", lens=(5, 16, 37), seed=7, **kw):
    return synth.build("t", num_seqs, Hq, Hkv, D, dtype, list(lens), seed, **kw)


# ---------------------------------------------------------------------------
# 16-bit decoders (library pins: numpy float16, torch bfloat16)
# ---------------------------------------------------------------------------
def test_decode_f16_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_bits(bits, "f16")
    want = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))


def test_decode_bf16_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_bits(bits, "bf16")
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


# ---------------------------------------------------------------------------
# the block-table figure (vLLM reading notes, section 核心思想)
# ---------------------------------------------------------------------------
def _page3():
    with open(os.path.join(GOLDEN, "page3_block_table.json")) as f:
        return json.load(f)


def test_page3_tables_match_pool_row():
    g = _page3()
    row = g["pool_row"]
    for req, table in g["tables"].items():
        # logical block i of request `req` is printed as "<req>-<i+1>" in the pool row
        from_row = [row.index(f"{req}-{i + 1}") for i in range(len(table))]
        assert from_row == table
    used = {b for t in g["tables"].values() for b in t}
    assert sorted(set(range(g["pool_blocks"])) - used) == g["free_blocks"]


def _tagged_pool(nblocks, Hkv=1, D=8):
    """Pool whose slot (b, o) holds the value b*16+o in every element (exact in fp16)."""
    tag = (np.arange(nblocks)[:, None] * 16 + np.arange(16)[None, :]).astype(np.float64)
    vals = np.broadcast_to(tag[:, None, :, None], (nblocks, Hkv, 16, D))
    return f16_bits(vals).copy()


def test_page3_gather_reads_the_printed_blocks():
    g = _page3()
    pool = _tagged_pool(g["pool_blocks"])
    tables = np.array([g["tables"]["A"], g["tables"]["B"]], dtype=np.int32)
    for s, req in enumerate(["A", "B"]):
        k, v = oracle.gather_kv(pool, pool, tables, s, 48)
        got = k[0, :, 0].view(np.float16).astype(int).tolist()
        want = [b * 16 + o for b in g["tables"][req] for o in range(16)]
        assert got == want
        assert np.array_equal(k, v)


def test_page3_decode_uses_the_tables():
    # all keys equal -> uniform weights -> output is the mean of A's (resp. B's) tags
    g = _page3()
    Hkv, D = 1, 8
    vpool = _tagged_pool(g["pool_blocks"], Hkv, D)
    kpool = f16_bits(np.zeros((g["pool_blocks"], Hkv, 16, D)))
    tables = np.array([g["tables"]["A"], g["tables"]["B"]], dtype=np.int32)
    q = f16_bits(np.ones((2, 1, D)))
    out = oracle.decode(q, kpool, vpool, tables, np.array([48, 40], np.int32), 0.125, "f16")
    for s, (req, L) in enumerate([("A", 48), ("B", 40)]):
        tags = [b * 16 + o for b in g["tables"][req] for o in range(16)][:L]
        assert np.all(out[s, 0] == math.fsum(tags) / L)


# ---------------------------------------------------------------------------
# KV size accounting (mlsys course page, section 6, 例 1)
# ---------------------------------------------------------------------------
def test_page5_kv_bytes_example():
    with open(os.path.join(GOLDEN, "page5_kv_bytes.json")) as f:
        g = json.load(f)
    got = synth.kv_bytes(g["tokens"], g["num_layers"], g["hidden"], g["bytes_per_element"])
    assert got == g["exact_bytes"] == 2 ** 30
    assert abs(got / 1e9 - g["printed_approx_gb"]) < 0.08


# ---------------------------------------------------------------------------
# library pin: identity-table paged attention == textbook attention
# ---------------------------------------------------------------------------
def _contiguous_case(rng, lens, Hq, Hkv, D, dtype):
    """Random K/V per sequence laid out on consecutive blocks (identity tables)."""
    nbs = [synth.cdiv(L, 16) for L in lens]
    nblocks = sum(nbs) + 1
    maxb = max(nbs)
    k = synth.to_bits(rng.standard_normal((nblocks, Hkv, 16, D)).astype(np.float32), dtype)
    v = synth.to_bits(rng.standard_normal((nblocks, Hkv, 16, D)).astype(np.float32), dtype)
    q = synth.to_bits(rng.standard_normal((len(lens), Hq, D)).astype(np.float32), dtype)
    tables = np.full((len(lens), maxb), -1, np.int32)
    b0 = 0
    for s, nb in enumerate(nbs):
        tables[s, :nb] = np.arange(b0, b0 + nb)
        b0 += nb
    return q, k, v, tables


@pytest.mark.parametrize("Hq,Hkv,D,dtype", [(4, 4, 16, "f16"), (8, 2, 32, "bf16"),
                                            (10, 2, 64, "f16"), (6, 2, 128, "bf16"),
                                            (5, 1, 64, "f16")])
def test_identity_table_equals_sdpa(Hq, Hkv, D, dtype):
    rng = np.random.default_rng(11)
    lens = [1, 15, 16, 17, 50]
    q, k, v, tables = _contiguous_case(rng, lens, Hq, Hkv, D, dtype)
    scale = 1.0 / math.sqrt(D)
    out = oracle.decode(q, k, v, tables, np.array(lens, np.int32), scale, dtype)
    kd = oracle.decode_bits(k, dtype)
    vd = oracle.decode_bits(v, dtype)
    qd = oracle.decode_bits(q, dtype)
    for s, L in enumerate(lens):
        blocks = tables[s, :synth.cdiv(L, 16)]
        # contiguous [Hkv, L, D] by concatenating the sequence's blocks
        kc = np.concatenate([kd[b] for b in blocks], axis=1)[:, :L]
        vc = np.concatenate([vd[b] for b in blocks], axis=1)[:, :L]
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(qd[s])[None, :, None, :], torch.from_numpy(kc)[None],
            torch.from_numpy(vc)[None], scale=scale, enable_gqa=True)[0, :, 0, :].numpy()
        np.testing.assert_allclose(out[s], ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# invariances and closed forms
# ---------------------------------------------------------------------------
def test_block_permutation_is_bit_exact():
    w = small(lens=(1, 17, 48, 100), num_seqs=4, pool_factor=2.0)
    base = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, w.dtype)
    perm = np.random.default_rng(3).permutation(w.num_blocks)
    k2 = np.empty_like(w.k_cache)
    v2 = np.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    t2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    out = oracle.decode(w.q, k2, v2, t2, w.seq_lens, w.scale, w.dtype)
    assert np.array_equal(out, base)


def test_seq_len_one_returns_v():
    w = small(lens=(1, 1, 1), dtype="bf16")
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, w.dtype)
    vd = oracle.decode_bits(w.v_cache, w.dtype)
    for s in range(3):
        for h in range(w.num_heads):
            assert np.array_equal(out[s, h], vd[w.block_tables[s, 0], h // w.group, 0])


def test_identical_keys_give_mean_of_v():
    w = small(lens=(3, 33, 64))
    k = w.k_cache.copy()
    k[:] = k[0, :, 0:1, :]          # one key vector per kv head, everywhere
    out = oracle.decode(w.q, k, w.v_cache, w.block_tables, w.seq_lens, w.scale, w.dtype)
    for s, L in enumerate(w.seq_lens):
        kv, vv = oracle.gather_kv(k, w.v_cache, w.block_tables, s, int(L))
        vd = oracle.decode_bits(vv, w.dtype)
        for h in range(w.num_heads):
            g = h // w.group
            mean = [math.fsum(vd[g, :, d]) / L for d in range(w.head_dim)]
            np.testing.assert_allclose(out[s, h], mean, rtol=0, atol=1e-14)


def test_scale_zero_gives_mean_of_v():
    w = small(lens=(7, 16, 31), scale=0.0)
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, 0.0, w.dtype)
    for s, L in enumerate(w.seq_lens):
        _, vv = oracle.gather_kv(w.k_cache, w.v_cache, w.block_tables, s, int(L))
        vd = oracle.decode_bits(vv, w.dtype)
        for h in range(w.num_heads):
            np.testing.assert_allclose(out[s, h], vd[h // w.group].mean(axis=0), rtol=0, atol=1e-14)


def test_token_order_does_not_matter():
    rng = np.random.default_rng(5)
    lens = [40, 23]
    q, k, v, tables = _contiguous_case(rng, lens, 4, 2, 16, "f16")
    base = oracle.decode(q, k, v, tables, np.array(lens, np.int32), 0.3, "f16")
    # move token slots around inside each sequence's blocks (K and V together)
    k2, v2 = k.copy(), v.copy()
    for s, L in enumerate(lens):
        pos = rng.permutation(L)
        for t_new, t_old in enumerate(pos):
            bn, on = tables[s, t_new // 16], t_new % 16
            bo, oo = tables[s, t_old // 16], t_old % 16
            k2[bn, :, on] = k[bo, :, oo]
            v2[bn, :, on] = v[bo, :, oo]
    out = oracle.decode(q, k2, v2, tables, np.array(lens, np.int32), 0.3, "f16")
    np.testing.assert_allclose(out, base, rtol=0, atol=1e-13)


def test_value_shift_moves_output():
    # softmax weights sum to one: o(V + c) = o(V) + c (integers keep fp16 exact)
    rng = np.random.default_rng(9)
    lens = [30, 9]
    q, k, _, tables = _contiguous_case(rng, lens, 2, 1, 16, "f16")
    vals = rng.integers(-8, 9, size=(k.shape[0], 1, 16, 16)).astype(np.float64)
    out0 = oracle.decode(q, k, f16_bits(vals), tables, np.array(lens, np.int32), 0.25, "f16")
    out1 = oracle.decode(q, k, f16_bits(vals + 16), tables, np.array(lens, np.int32), 0.25, "f16")
    np.testing.assert_allclose(out1, out0 + 16, rtol=0, atol=1e-12)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(4)
    lens = [20]
    D = 16
    q, k, v, tables = _contiguous_case(rng, lens, 1, 1, D, "f16")
    qv = np.zeros(D); qv[3] = 4.0
    q = f16_bits(qv[None, None, :])
    kd = np.zeros((k.shape[0], 1, 16, D))
    t_star = 13
    kd[tables[0, t_star // 16], 0, t_star % 16, 3] = 64.0      # score 256 vs 0
    out = oracle.decode(q, f16_bits(kd), v, tables, np.array(lens, np.int32), 1.0, "f16")
    vd = oracle.decode_bits(v, "f16")[tables[0, 0], 0, t_star]
    np.testing.assert_allclose(out[0, 0], vd, rtol=0, atol=1e-100)


def test_nan_in_unreached_slots_changes_nothing():
    w0 = small(lens=(3, 17, 33), num_seqs=3)
    w1 = small(lens=(3, 17, 33), num_seqs=3, poison=True)
    o0 = oracle.decode(w0.q, w0.k_cache, w0.v_cache, w0.block_tables, w0.seq_lens, w0.scale, "f16")
    o1 = oracle.decode(w1.q, w1.k_cache, w1.v_cache, w1.block_tables, w1.seq_lens, w1.scale, "f16")
    assert np.isfinite(o1).all()
    assert np.array_equal(o0, o1)


def test_empty_sequence_gives_zeros():
    w = small(lens=(0, 5, 0))
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, w.dtype)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)


# ---------------------------------------------------------------------------
# brute force on tiny inputs
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("Hq,Hkv,dtype", [(2, 2, "f16"), (4, 2, "bf16"), (6, 2, "f16"),
                                          (3, 1, "bf16")])
def test_brute_force_agrees(Hq, Hkv, dtype):
    w = small(num_seqs=4, Hq=Hq, Hkv=Hkv, D=8, dtype=dtype, lens=(0, 1, 17, 33), seed=21)
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, dtype)
    ref = brute.paged_attention(w.q.tolist(), w.k_cache.tolist(), w.v_cache.tolist(),
                                w.block_tables.tolist(), w.seq_lens.tolist(), w.scale, dtype)
    np.testing.assert_allclose(out, np.array(ref), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# split-K partials and the log-sum-exp merge
# ---------------------------------------------------------------------------
def test_partials_merge_back_to_decode():
    w = small(lens=(5, 96, 130, 200), num_seqs=4, Hq=4, Hkv=2, D=16)
    P = 32
    m, l, o = oracle.partials(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                              w.scale, w.dtype, P)
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, w.dtype)
    for s, L in enumerate(w.seq_lens):
        n = synth.cdiv(int(L), P)
        assert np.all(l[s, :, n:] == 0)
        for h in range(w.num_heads):
            merged = oracle.lse_merge(m[s, h, :n], l[s, h, :n], o[s, h, :n])
            np.testing.assert_allclose(merged, out[s, h], rtol=0, atol=1e-12)


def test_single_partition_is_the_decode():
    w = small(lens=(5, 31, 60))
    m, l, o = oracle.partials(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                              w.scale, w.dtype, 64)
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, w.dtype)
    assert np.array_equal(o[:, :, 0], out)
    assert np.array_equal(oracle.lse_merge(m[0, 0, :1], l[0, 0, :1], o[0, 0, :1]), out[0, 0])


def test_partial_m_and_l_definitions():
    w = small(lens=(70,), num_seqs=1, Hq=2, Hkv=1, D=8)
    P = 32
    m, l, _ = oracle.partials(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                              w.scale, w.dtype, P)
    kk, _ = oracle.gather_kv(w.k_cache, w.v_cache, w.block_tables, 0, 70)
    kd = oracle.decode_bits(kk, "f16")[0]
    for h in range(2):
        qd = oracle.decode_bits(w.q[0, h], "f16")
        x = [w.scale * math.fsum(qd * kd[t]) for t in range(70)]
        for p in range(3):
            seg = x[p * P:(p + 1) * P]
            assert abs(m[0, h, p] - max(seg)) < 1e-13
            assert abs(l[0, h, p] - math.fsum(math.exp(a - max(seg)) for a in seg)) < 1e-12


def test_lse_merge_closed_form():
    o1 = np.arange(4.0)
    o2 = np.arange(4.0) * -2 + 1
    # weights l_p * exp(m_p - M): 1 and 3
    got = oracle.lse_merge([0.0, math.log(3.0)], [1.0, 1.0], np.stack([o1, o2]))
    np.testing.assert_allclose(got, (o1 + 3 * o2) / 4, rtol=0, atol=1e-15)
    # an empty partial carries no weight
    got = oracle.lse_merge([5.0, -np.inf], [2.0, 0.0], np.stack([o1, o2]))
    assert np.array_equal(got, o1)


# ---------------------------------------------------------------------------
# pool maintenance: reshape_and_cache and copy_blocks
# ---------------------------------------------------------------------------
def test_reshape_and_cache_writes_only_the_slots():
    w = synth.tiny()
    k, v = w.k_cache.copy(), w.v_cache.copy()
    slots = w.slot_mapping.copy()
    slots[1] = -1                                  # padding token: skipped
    bad = oracle.reshape_and_cache(k, v, w.k_new, w.v_new, slots)
    assert bad == 0
    changed = np.zeros(k.shape[:1] + k.shape[2:3], dtype=bool)
    for s, L in enumerate(w.seq_lens):
        kk, vv = oracle.gather_kv(k, v, w.block_tables, s, int(L))
        if s == 1:
            ko, _ = oracle.gather_kv(w.k_cache, w.v_cache, w.block_tables, s, int(L))
            assert np.array_equal(kk, ko)
            continue
        assert np.array_equal(kk[:, -1], w.k_new[s]) and np.array_equal(vv[:, -1], w.v_new[s])
        changed[slots[s] // 16, slots[s] % 16] = True
    diff = (k != w.k_cache).any(axis=(1, 3)) | (v != w.v_cache).any(axis=(1, 3))
    assert not (diff & ~changed).any()


def test_reshape_and_cache_counts_slots_past_the_pool():
    w = synth.tiny()
    k, v = w.k_cache.copy(), w.v_cache.copy()
    slots = w.slot_mapping.copy()
    slots[0] = w.num_blocks * 16
    assert oracle.reshape_and_cache(k, v, w.k_new, w.v_new, slots) == 1


def test_copy_blocks_copies_whole_blocks():
    w = synth.parsamp(num_prompts=2, samples=4, prompt_len=40, max_suffix=20,
                      num_heads=4, num_kv_heads=2, head_dim=16)
    k, v = w.k_cache.copy(), w.v_cache.copy()
    assert oracle.copy_blocks(k, v, w.block_mapping) == 0
    dsts = set()
    for src, dst in w.block_mapping:
        assert np.array_equal(k[dst], w.k_cache[src]) and np.array_equal(v[dst], w.v_cache[src])
        dsts.add(int(dst))
    others = np.array([b not in dsts for b in range(w.num_blocks)])
    assert np.array_equal(k[others], w.k_cache[others])
    bad = np.array([[0, w.num_blocks]], np.int64)
    assert oracle.copy_blocks(k, v, bad) == 1


# ---------------------------------------------------------------------------
# copy-on-write and shared prefixes (parallel sampling)
# ---------------------------------------------------------------------------
def test_cow_remap_keeps_outputs_bit_exact():
    # block-aligned prompt: the remapped block is a byte copy, outputs are identical
    w = synth.parsamp(num_prompts=2, samples=4, prompt_len=64, max_suffix=20,
                      num_heads=4, num_kv_heads=2, head_dim=16)
    k, v = w.k_cache.copy(), w.v_cache.copy()
    oracle.reshape_and_cache(k, v, w.k_new, w.v_new, w.slot_mapping)
    before = oracle.decode(w.q, k, v, w.tables_before_cow, w.seq_lens, w.scale, w.dtype)
    oracle.copy_blocks(k, v, w.block_mapping)
    after = oracle.decode(w.q, k, v, w.block_tables, w.seq_lens, w.scale, w.dtype)
    assert np.array_equal(before, after)


def test_cow_unaligned_prefix_has_no_crosstalk():
    # unaligned prompt, zero suffix: every sample's new token lands in its own copy of
    # the shared partial block; changing one sample's token moves only its output
    kw = dict(num_prompts=1, samples=4, prompt_len=40, suffix_lens=[0, 0, 0, 0],
              num_heads=4, num_kv_heads=2, head_dim=16)
    w = synth.parsamp(poison=True, **kw)
    out0, _, _ = oracle.step(w)
    assert np.isfinite(out0).all()
    w.k_new = w.k_new.copy()
    w.k_new[2] = synth.to_bits(np.full(w.k_new[2].shape, 3.0, np.float32), "f16")
    out1, _, _ = oracle.step(w)
    changed = [not np.array_equal(out0[s], out1[s]) for s in range(4)]
    assert changed == [False, False, True, False]


# ---------------------------------------------------------------------------
# the synthetic workloads themselves
# ---------------------------------------------------------------------------
def test_workload_shapes():
    t = synth.tiny()
    assert t.num_blocks == 64 and t.seq_lens.min() >= 1 and t.seq_lens.max() <= 100
    assert t.k_new.shape == (4, 8, 64)
    assert synth.kv_bytes(sum(synth.LONG_LENS), 1, 8 * 128, 2) == 1342177280
    lens = synth.lens_gqa8b(np.random.default_rng(1003), 100000)
    assert lens.min() == 16 and lens.max() == 4096
    assert 500 < np.median(lens) < 700
    p = synth.parsamp(num_heads=4, num_kv_heads=1, head_dim=64)
    assert p.block_mapping.shape == (112, 2) and p.num_seqs == 128
    assert p.seq_lens.min() >= 1025 and p.seq_lens.max() <= 1024 + 256 + 1


def test_swap_out_and_back_restores_blocks():
    # preemption by swapping (OS-paging table): blocks go to a host pool and come back
    w = synth.build("swap", 6, 16, 4, 64, "bf16", [40, 100, 300, 17, 64, 5], seed=8,
                    pool_factor=3.0)
    rng = np.random.default_rng(2)
    seq_blocks = w.block_tables[2, :synth.cdiv(int(w.seq_lens[2]), 16)]
    host_k = np.zeros((len(seq_blocks) + 3,) + w.k_cache.shape[1:], np.uint16)
    host_v = np.zeros_like(host_k)
    out_pairs = np.stack([seq_blocks, 3 + np.arange(len(seq_blocks))], 1).astype(np.int64)
    assert oracle.swap_blocks(host_k, host_v, w.k_cache, w.v_cache, out_pairs) == 0
    for src, dst in out_pairs:
        assert np.array_equal(host_k[dst], w.k_cache[src]) and np.array_equal(host_v[dst], w.v_cache[src])
    assert not host_k[:3].any()                           # untouched host blocks stay as they were
    # back into other device blocks: decode through the remapped table is unchanged
    free = np.setdiff1d(np.arange(w.num_blocks), w.block_tables[w.block_tables >= 0])
    new_ids = rng.choice(free, size=len(seq_blocks), replace=False)
    k2, v2 = w.k_cache.copy(), w.v_cache.copy()
    in_pairs = np.stack([3 + np.arange(len(seq_blocks)), new_ids], 1).astype(np.int64)
    assert oracle.swap_blocks(k2, v2, host_k, host_v, in_pairs) == 0
    t2 = w.block_tables.copy()
    t2[2, :len(seq_blocks)] = new_ids
    base = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, w.dtype)
    again = oracle.decode(w.q, k2, v2, t2, w.seq_lens, w.scale, w.dtype)
    assert np.array_equal(base, again)
    assert oracle.swap_blocks(k2, v2, host_k, host_v, np.array([[0, w.num_blocks]])) == 1


# ---------------------------------------------------------------------------
# chunked prefill (causal attention of a chunk of new tokens over the pool)
# ---------------------------------------------------------------------------
def _prefill_case(dtype="f16", Hq=8, Hkv=2, D=32):
    return synth.build_prefill("pf", Hq, Hkv, D, dtype, [5, 40, 70, 16], [5, 17, 33, 1], seed=31)


def test_prefill_rows_are_decodes_of_their_prefixes():
    w = _prefill_case()
    out = oracle.prefill(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.query_start,
                         w.scale, w.dtype)
    for s in range(w.num_seqs):
        c = w.query_start[s + 1] - w.query_start[s]
        for i in range(c):
            row = w.query_start[s] + i
            p = int(w.seq_lens[s]) - c + i
            one = oracle.decode(w.q[row][None], w.k_cache, w.v_cache, w.block_tables[s][None],
                                np.array([p + 1], np.int32), w.scale, w.dtype)
            assert np.array_equal(out[row], one[0])


@pytest.mark.parametrize("Hq,Hkv,D,dtype", [(4, 4, 16, "f16"), (8, 2, 64, "bf16")])
def test_prefill_equals_causal_sdpa(Hq, Hkv, D, dtype):
    rng = np.random.default_rng(12)
    lens, chunks = [30, 64, 9], [30, 20, 4]
    q_, k, v, tables = _contiguous_case(rng, lens, Hq, Hkv, D, dtype)
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = synth.to_bits(rng.standard_normal((qs[-1], Hq, D)).astype(np.float32), dtype)
    scale = 1.0 / math.sqrt(D)
    out = oracle.prefill(q, k, v, tables, np.array(lens, np.int32), qs, scale, dtype)
    kd, vd, qd = (oracle.decode_bits(x, dtype) for x in (k, v, q))
    for s, (L, c) in enumerate(zip(lens, chunks)):
        blocks = tables[s, :synth.cdiv(L, 16)]
        kc = np.concatenate([kd[b] for b in blocks], axis=1)[:, :L]
        vc = np.concatenate([vd[b] for b in blocks], axis=1)[:, :L]
        # chunk row i (position L-c+i) may see tokens 0..L-c+i
        mask = np.arange(L)[None, :] <= (L - c + np.arange(c))[:, None]
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(qd[qs[s]:qs[s + 1]]).permute(1, 0, 2)[None],
            torch.from_numpy(kc)[None], torch.from_numpy(vc)[None],
            attn_mask=torch.from_numpy(mask), scale=scale, enable_gqa=True)[0].permute(1, 0, 2)
        np.testing.assert_allclose(out[qs[s]:qs[s + 1]], ref.numpy(), rtol=0, atol=1e-12)
