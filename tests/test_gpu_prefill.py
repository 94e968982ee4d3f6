"""GPU parity of pa_prefill (tcgen05 chunked-prefill attention) against the
fp64 oracle: ragged chunks over ragged contexts, every supported head size,
both dtypes, GQA groups that do and do not divide the 128-row tile, pools
poisoned with NaN outside live tokens, empty chunks, whole-prompt chunks, and
the error paths.  At the full prefill workload, sampled rows are checked
against the oracle's decode of the row's prefix (equal to its prefill row,
which the oracle tests pin)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, TORCH_DTYPE, dev_bits, max_err

pytestmark = pytest.mark.gpu


def _run(pa, w, max_query_len=None, tables=None):
    q = dev_bits(w.q, w.dtype)
    k, v = dev_bits(w.k_cache, w.dtype), dev_bits(w.v_cache, w.dtype)
    out = torch.full_like(q, float("nan"))
    qs = torch.from_numpy(w.query_start).cuda()
    t = torch.from_numpy(w.block_tables if tables is None else tables).cuda()
    mq = int(np.diff(w.query_start).max()) if max_query_len is None else max_query_len
    pa.prefill(out, q, k, v, t, torch.from_numpy(w.seq_lens).cuda(), qs, mq, w.scale)
    return out


def _ref(w):
    return oracle.prefill(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.query_start,
                          w.scale, w.dtype)


CASES = [
    # Hq, Hkv, D, dtype, seq_lens, chunk_lens
    (8, 2, 128, "bf16", [300, 70, 129, 1000, 64, 17], [300, 33, 1, 200, 64, 5]),
    (8, 8, 64, "f16", [40, 257, 511, 96], [40, 150, 77, 96]),
    (32, 4, 128, "f16", [700, 65, 33], [140, 65, 20]),
    (16, 16, 128, "bf16", [130, 1], [130, 1]),
    (12, 4, 64, "bf16", [250, 90, 400], [250, 43, 61]),      # G = 3: 42 tokens, 2 idle rows
    (32, 2, 128, "bf16", [500, 200], [97, 200]),             # G = 16: 8 tokens per block
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_prefill_matches_oracle(pa, case):
    hq, hkv, d, dt, lens, chunks = CASES[case]
    w = synth.build_prefill("pf", hq, hkv, d, dt, lens, chunks, seed=40 + case, poison=True)
    out = _run(pa, w)
    assert pa.get_device_error() == 0
    assert max_err(out, _ref(w)) <= TOL[dt]


def test_prefill_empty_chunks_and_untouched_rows(pa):
    w = synth.build_prefill("pf", 8, 2, 128, "f16", [50, 80, 30, 200], [0, 80, 0, 64], seed=9,
                            poison=True)
    out = _run(pa, w)
    assert pa.get_device_error() == 0
    assert out.shape[0] == 144
    assert max_err(out, _ref(w)) <= TOL["f16"]


def test_prefill_chunk_longer_than_max_query_len_is_reported(pa):
    w = synth.build_prefill("pf", 8, 2, 64, "bf16", [300, 100], [300, 40], seed=5)
    _run(pa, w, max_query_len=100)       # 300 rows do not fit 100
    assert pa.get_device_error() & pa.DEVERR["QUERY_RANGE"]
    w2 = synth.build_prefill("pf", 8, 2, 64, "bf16", [30, 100], [30, 40], seed=5)
    w2.seq_lens[0] = 20                  # chunk of 30 longer than its sequence
    out = _run(pa, w2)
    assert pa.get_device_error() == pa.DEVERR["QUERY_RANGE"]
    ref = _ref_rows(w2, 1)
    assert max_err(out[30:], ref) <= TOL["bf16"]


def _ref_rows(w, s):
    qs = w.query_start
    return oracle.prefill(w.q[qs[s]:qs[s + 1]], w.k_cache, w.v_cache, w.block_tables[s:s + 1],
                          w.seq_lens[s:s + 1], np.array([0, qs[s + 1] - qs[s]], np.int32),
                          w.scale, w.dtype)


def test_prefill_bad_table_entry_is_reported(pa):
    w = synth.build_prefill("pf", 8, 2, 128, "f16", [100, 60], [30, 60], seed=6)
    tables = w.block_tables.copy()
    tables[0, 2] = w.num_blocks + 5
    _run(pa, w, tables=tables)
    assert pa.get_device_error() == pa.DEVERR["TABLE_RANGE"]


def test_prefill_full_workload_sampled_rows(pa):
    # the 8 x 512-token chunk workload; 3 rows of every sequence and all heads
    # checked against the oracle's decode of the row's prefix
    w = synth.prefill_chunks()
    out = _run(pa, w)
    assert pa.get_device_error() == 0
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    rng = np.random.default_rng(3)
    for s in range(w.num_seqs):
        c = int(w.query_start[s + 1] - w.query_start[s])
        for i in sorted(set([0, c - 1, int(rng.integers(c))])):
            row = int(w.query_start[s]) + i
            p = int(w.seq_lens[s]) - c + i
            ref = oracle.decode(w.q[row][None], w.k_cache, w.v_cache, w.block_tables[s][None],
                                np.array([p + 1], np.int32), w.scale, w.dtype)
            assert float(np.abs(got[row] - ref[0]).max()) <= TOL[w.dtype], (s, i)


def test_prefill_then_decode_continues_the_sequence(pa):
    # a prompt prefilled in two chunks, then one decode step; each stage
    # against the oracle on the same pool
    rng = np.random.default_rng(2)
    hq, hkv, d, dt = 8, 2, 128, "bf16"
    nb, L1, L2 = 32, 70, 45
    k_host = synth.to_bits(rng.standard_normal((nb, hkv, 16, d)).astype(np.float32), dt)
    v_host = synth.to_bits(rng.standard_normal((nb, hkv, 16, d)).astype(np.float32), dt)
    k_dev, v_dev = dev_bits(k_host, dt), dev_bits(v_host, dt)
    table = rng.permutation(nb)[:8].astype(np.int32)[None]
    tab_d = torch.from_numpy(table).cuda()
    scale = d ** -0.5
    done = 0
    for c in (L1, L2):
        kn = synth.to_bits(rng.standard_normal((c, hkv, d)).astype(np.float32), dt)
        vn = synth.to_bits(rng.standard_normal((c, hkv, d)).astype(np.float32), dt)
        pos = done + np.arange(c)
        slots = (table[0][pos // 16].astype(np.int64) * 16 + pos % 16)
        pa.reshape_and_cache(dev_bits(kn, dt), dev_bits(vn, dt), k_dev, v_dev,
                             torch.from_numpy(slots).cuda())
        oracle.reshape_and_cache(k_host, v_host, kn, vn, slots)
        done += c
        q = synth.to_bits(rng.standard_normal((c, hq, d)).astype(np.float32), dt)
        qd = dev_bits(q, dt)
        out = torch.empty_like(qd)
        lens = np.array([done], np.int32)
        qs = np.array([0, c], np.int32)
        pa.prefill(out, qd, k_dev, v_dev, tab_d, torch.from_numpy(lens).cuda(),
                   torch.from_numpy(qs).cuda(), c, scale)
        ref = oracle.prefill(q, k_host, v_host, table, lens, qs, scale, dt)
        assert max_err(out, ref) <= TOL[dt]
    q = synth.to_bits(rng.standard_normal((1, hq, d)).astype(np.float32), dt)
    out = torch.empty(1, hq, d, dtype=TORCH_DTYPE[dt], device="cuda")
    pa.decode(out, dev_bits(q, dt), k_dev, v_dev, tab_d,
              torch.tensor([done], dtype=torch.int32, device="cuda"), scale)
    ref = oracle.decode(q, k_host, v_host, table, np.array([done], np.int32), scale, dt)
    assert max_err(out, ref) <= TOL[dt]
    assert pa.get_device_error() == 0


def test_prefill_work_order_does_not_change_results(pa):
    # with the planning workspace (longest work first) and without it, the
    # output is bit-identical; a too-small workspace is refused
    w = synth.build_prefill("pf", 32, 8, 128, "bf16", [900, 130, 2000, 64, 700],
                            [600, 130, 200, 1, 333], seed=21, poison=True)
    q = dev_bits(w.q, w.dtype)
    k, v = dev_bits(w.k_cache, w.dtype), dev_bits(w.v_cache, w.dtype)
    t = torch.from_numpy(w.block_tables).cuda()
    lens = torch.from_numpy(w.seq_lens).cuda()
    qs = torch.from_numpy(w.query_start).cuda()
    mq = int(np.diff(w.query_start).max())
    a, b = torch.empty_like(q), torch.empty_like(q)
    pa.prefill(a, q, k, v, t, lens, qs, mq, w.scale, workspace=None)
    pa.prefill(b, q, k, v, t, lens, qs, mq, w.scale)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert pa.get_device_error() == 0
    assert max_err(a, _ref(w)) <= TOL["bf16"]
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PagedAttnError) as e:
        pa.prefill(b, q, k, v, t, lens, qs, mq, w.scale, workspace=small)
    assert e.value.status == 3


def test_prefill_in_a_cuda_graph(pa):
    # the planning kernel and the dependent prefill launch are captured and
    # replayed; replays match the eager call bit for bit
    w = synth.build_prefill("pf", 32, 8, 128, "bf16", [700, 300, 1200], [300, 300, 64], seed=23)
    q = dev_bits(w.q, w.dtype)
    k, v = dev_bits(w.k_cache, w.dtype), dev_bits(w.v_cache, w.dtype)
    t = torch.from_numpy(w.block_tables).cuda()
    lens = torch.from_numpy(w.seq_lens).cuda()
    qs = torch.from_numpy(w.query_start).cuda()
    mq = int(np.diff(w.query_start).max())
    ws = torch.empty(pa.prefill_workspace_size(w.num_seqs, mq, w.num_heads, w.num_kv_heads),
                     dtype=torch.uint8, device="cuda")
    eager, out = torch.empty_like(q), torch.zeros_like(q)
    pa.prefill(eager, q, k, v, t, lens, qs, mq, w.scale, workspace=ws)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pa.prefill(out, q, k, v, t, lens, qs, mq, w.scale, workspace=ws, stream=s)   # warm-up
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pa.prefill(out, q, k, v, t, lens, qs, mq, w.scale, workspace=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert pa.get_device_error() == 0


def test_prefill_of_single_token_chunks_is_a_decode(pa):
    # 200 sequences whose chunk is their newest token: the prefill is a
    # decode batch; both kernels agree with the oracle's decode
    rng = np.random.default_rng(8)
    lens = rng.integers(1, 900, size=200)
    w = synth.build_prefill("pf", 32, 8, 128, "bf16", lens, np.ones(200, int), seed=24, poison=True)
    out = _run(pa, w)
    assert pa.get_device_error() == 0
    ref = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, w.dtype)
    assert max_err(out, ref) <= TOL["bf16"]
    dec = torch.empty_like(out)
    pa.decode(dec, dev_bits(w.q, w.dtype), dev_bits(w.k_cache, w.dtype),
              dev_bits(w.v_cache, w.dtype), torch.from_numpy(w.block_tables).cuda(),
              torch.from_numpy(w.seq_lens).cuda(), w.scale)
    assert max_err(dec, ref) <= TOL["bf16"]


def test_prefill_long_prompt_sampled_rows(pa):
    # an 8192-token prompt prefilled as one chunk (64 blocks of 256 rows per
    # kv head), plus a 2048-token chunk over 14000 tokens of context; rows
    # sampled along the chunk against the oracle's decode of their prefix
    w = synth.build_prefill("pf", 16, 4, 128, "f16", [8192, 16048], [8192, 2048], seed=25)
    out = _run(pa, w)
    assert pa.get_device_error() == 0
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    for s in range(w.num_seqs):
        c = int(w.query_start[s + 1] - w.query_start[s])
        for i in (0, 1, 127, 128, 129, c // 2, c - 257, c - 2, c - 1):
            row = int(w.query_start[s]) + i
            p = int(w.seq_lens[s]) - c + i
            ref = oracle.decode(w.q[row][None], w.k_cache, w.v_cache, w.block_tables[s][None],
                                np.array([p + 1], np.int32), w.scale, w.dtype)
            assert float(np.abs(got[row] - ref[0]).max()) <= TOL["f16"], (s, i)



@pytest.mark.parametrize("dt,every,step,d", [("bf16", 64, 10.0, 128), ("bf16", 128, 6.5, 128),
                                             ("f16", 64, 10.0, 128), ("bf16", 64, 10.0, 64)])
def test_prefill_scores_that_keep_growing(pa, dt, every, step, d):
    # Every query row leans along one direction u, and every `every`-th key
    # (at offset 37, so the spikes fall in both halves of 128-key tiles when
    # every = 64) lies along u with a length that raises its score by about
    # `step` natural-log units over the previous spike.  Each row's running
    # maximum therefore keeps rising past the kernel's lazy-rescale
    # threshold (2^8), inside tiles and at their boundaries, and the result
    # depends on the rescale of O, of the row sum and of P already written.
    # The keys are aligned with the queries, so the large scores carry no
    # cancellation; V is scaled by 1/4 so that |O| stays near 1 and the
    # dtype's tolerance (derived for outputs of that size) applies.
    w = synth.build_prefill("pf", 8, 2, d, dt, [700, 300, 1000, 129], [300, 300, 200, 129],
                            seed=77, poison=True)
    rng = np.random.default_rng(78)
    u = rng.standard_normal(d)
    u /= np.linalg.norm(u)
    beta = 3.0
    q = dev_bits(w.q, dt, device="cpu").float().numpy() + (beta * u).astype(np.float32)
    w.q = synth.to_bits(q, dt)
    k = dev_bits(w.k_cache, dt, device="cpu").float().numpy()
    v = dev_bits(w.v_cache, dt, device="cpu").float().numpy()
    for s in range(w.num_seqs):
        for p in range(int(w.seq_lens[s])):
            b, r = w.block_tables[s, p // 16], p % 16
            v[b, :, r, :] *= 0.25
            if p % every == 37 % every:
                target = 4.0 + step * (p // every)          # score of the spike, natural log units
                k[b, :, r, :] = (target / (beta * w.scale) * u).astype(np.float32)
    w.k_cache, w.v_cache = synth.to_bits(k, dt), synth.to_bits(v, dt)
    out = _run(pa, w)
    assert pa.get_device_error() == 0
    assert max_err(out, _ref(w)) <= TOL[dt]


HEADS = [(8, 8), (16, 8), (24, 8), (32, 8), (40, 8), (12, 4), (64, 4), (32, 2), (16, 1)]


@pytest.mark.parametrize("seed", range(12))
def test_prefill_random_shapes(pa, seed):
    # seeded sweep: head layout (G = 1, 2, 3, 4, 5, 16), head size, dtype,
    # 1-5 sequences of 1-700 tokens whose chunk is empty, one token, the whole
    # prompt or a random length; NaN-poisoned pools
    rng = np.random.default_rng(900 + seed)
    hq, hkv = HEADS[rng.integers(len(HEADS))]
    d = int(rng.choice([64, 128]))
    dt = str(rng.choice(["f16", "bf16"]))
    n = int(rng.integers(1, 6))
    lens = rng.integers(1, 701, size=n)
    lens[rng.random(n) < 0.2] = rng.integers(1, 17)          # some sequences shorter than a block
    kind = rng.integers(0, 4, size=n)
    chunks = np.where(kind == 0, 0, np.where(kind == 1, 1, np.where(kind == 2, lens,
                                                                     rng.integers(1, lens + 1))))
    if chunks.sum() == 0:
        chunks[0] = lens[0]
    w = synth.build_prefill("pf", hq, hkv, d, dt, lens, chunks, seed=1000 + seed, poison=True)
    out = _run(pa, w)
    assert pa.get_device_error() == 0
    assert max_err(out, _ref(w)) <= TOL[dt], (hq, hkv, d, dt, lens.tolist(), chunks.tolist())


def test_prefill_on_two_streams(pa):
    # two different prefills in flight on two side streams, each with its
    # own automatically allocated work-order workspace
    ws = [synth.build_prefill("pf", 16, 4, 128, "bf16", [700, 300], [400, 300], seed=31, poison=True),
          synth.build_prefill("pf", 8, 8, 64, "f16", [90, 1000, 17], [90, 64, 17], seed=32, poison=True)]
    outs, streams = [], [torch.cuda.Stream(), torch.cuda.Stream()]
    args = []
    for w in ws:
        q = dev_bits(w.q, w.dtype)
        args.append((q, dev_bits(w.k_cache, w.dtype), dev_bits(w.v_cache, w.dtype),
                     torch.from_numpy(w.block_tables).cuda(), torch.from_numpy(w.seq_lens).cuda(),
                     torch.from_numpy(w.query_start).cuda(), int(np.diff(w.query_start).max())))
        outs.append(torch.full_like(q, float("nan")))
    torch.cuda.synchronize()
    for w, s, out, (q, k, v, t, lens, qs, mq) in zip(ws, streams, outs, args):
        with torch.cuda.stream(s):
            pa.prefill(out, q, k, v, t, lens, qs, mq, w.scale, stream=s)
    for s in streams:
        s.synchronize()
    assert pa.get_device_error() == 0
    for w, out in zip(ws, outs):
        assert max_err(out, _ref(w)) <= TOL[w.dtype]


def test_prefill_work_order_by_sequence_when_kv_exceeds_l2(pa):
    # six 8192-token contexts over 8 kv heads hold ~200 MB of K/V, more than
    # L2, so the work order keeps each sequence's tiles together; the output
    # is bit-identical to the fixed order and matches the oracle's decode of
    # each sampled row's prefix
    w = synth.build_prefill("pf", 32, 8, 128, "bf16", [8192] * 6, [300, 64, 1, 512, 129, 1000],
                            seed=61)
    q = dev_bits(w.q, w.dtype)
    k, v = dev_bits(w.k_cache, w.dtype), dev_bits(w.v_cache, w.dtype)
    t = torch.from_numpy(w.block_tables).cuda()
    lens = torch.from_numpy(w.seq_lens).cuda()
    qs = torch.from_numpy(w.query_start).cuda()
    mq = int(np.diff(w.query_start).max())
    a, b = torch.empty_like(q), torch.empty_like(q)
    pa.prefill(a, q, k, v, t, lens, qs, mq, w.scale, workspace=None)
    pa.prefill(b, q, k, v, t, lens, qs, mq, w.scale)
    assert pa.get_device_error() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    got = b.float().cpu().numpy().astype(np.float64)
    for s in range(w.num_seqs):
        c = int(w.query_start[s + 1] - w.query_start[s])
        for i in sorted({0, c // 3, c // 2, c - 1}):
            row = int(w.query_start[s]) + i
            p = int(w.seq_lens[s]) - c + i
            ref = oracle.decode(w.q[row][None], w.k_cache, w.v_cache, w.block_tables[s][None],
                                np.array([p + 1], np.int32), w.scale, w.dtype)
            assert float(np.abs(got[row] - ref[0]).max()) <= TOL["bf16"], (s, i)


def _plan_after(pa, w):
    """Run a prefill with an explicit work-order workspace and read the plan
    back: the pair count at byte 0, then one uint32 (sequence << 16 | query
    tile) per pair from byte 16."""
    q = dev_bits(w.q, w.dtype)
    k, v = dev_bits(w.k_cache, w.dtype), dev_bits(w.v_cache, w.dtype)
    mq = int(np.diff(w.query_start).max())
    nb = pa.prefill_workspace_size(w.num_seqs, mq, w.num_heads, w.num_kv_heads)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    pa.prefill(out, q, k, v, torch.from_numpy(w.block_tables).cuda(),
               torch.from_numpy(w.seq_lens).cuda(), torch.from_numpy(w.query_start).cuda(), mq,
               w.scale, workspace=ws)
    torch.cuda.synchronize()
    raw = ws.cpu().numpy()
    count = int(raw[:4].view(np.int32)[0])
    plan = raw[16:16 + 4 * count].view(np.uint32)
    return [(int(e >> 16), int(e & 0xFFFF)) for e in plan]


def _tile_counts(w):
    # key tiles (128 keys) up to the last row of each (sequence, query tile):
    # the query tile holds 2 * (128 / G) chunk tokens
    tpb = 2 * (128 // (w.num_heads // w.num_kv_heads))
    nt = {}
    for s in range(w.num_seqs):
        L = int(w.seq_lens[s])
        c = int(w.query_start[s + 1] - w.query_start[s])
        for t in range((c + tpb - 1) // tpb):
            nt[(s, t)] = (L - c + min((t + 1) * tpb, c) - 1) // 128 + 1
    return nt


def test_prefill_work_order_contents(pa):
    # the plan holds every (sequence, query tile) pair exactly once; a batch
    # whose K/V fits in L2 is ordered longest first, a larger one sequence by
    # sequence (sequences by their heaviest tile, each sequence's tiles
    # heaviest first)
    small = synth.build_prefill("pf", 32, 8, 128, "bf16", [900, 130, 2000, 64, 700],
                                [600, 130, 200, 1, 333], seed=21)
    plan, nt = _plan_after(pa, small), _tile_counts(small)
    assert sorted(plan) == sorted(nt)
    counts = [nt[e] for e in plan]
    assert counts == sorted(counts, reverse=True)

    big = synth.build_prefill("pf", 32, 8, 128, "bf16", [8192, 4096, 8192, 6000, 8192, 7000],
                              [300, 64, 1, 512, 129, 1000], seed=61)
    plan, nt = _plan_after(pa, big), _tile_counts(big)
    assert sorted(plan) == sorted(nt)
    seqs = [s for s, _ in plan]
    runs = [s for i, s in enumerate(seqs) if i == 0 or s != seqs[i - 1]]
    assert len(runs) == len(set(runs))                     # each sequence's pairs together
    heaviest = [max(nt[(s, t)] for (s2, t) in nt if s2 == s) for s in runs]
    assert heaviest == sorted(heaviest, reverse=True)
    for s in runs:
        tiles = [t for s2, t in plan if s2 == s]
        assert tiles == sorted(tiles, reverse=True)
    assert pa.get_device_error() == 0
