"""The rows working together the way an engine drives them: the host block
manager hands out slots; each prompt is prefilled in chunks (its K/V written
by reshape_and_cache, then the chunk attends through pa_prefill); one
sequence is forked into samples; decode steps follow, with the manager's
copy-on-write pairs going to copy_blocks and each new token's slot to
pa_decode_append.  Every stage is checked against the oracle run on a host
replica of the pool, and the pools end bit-identical."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, TORCH_DTYPE, dev_bits, host_bits, max_err
from paged_kv_cache_260_gb300.block_manager import BlockManager

pytestmark = pytest.mark.gpu


def test_chunked_prefill_then_forked_decode(pa):
    rng = np.random.default_rng(77)
    NB, HKV, HQ, D, MAXB, CHUNK = 160, 2, 8, 128, 24, 100
    dt = "bf16"
    scale = D ** -0.5

    def bits(*shape):
        return synth.to_bits(rng.standard_normal(shape).astype(np.float32), dt)

    k_host = bits(NB, HKV, 16, D)                            # stale contents everywhere
    v_host = bits(NB, HKV, 16, D)
    k_dev, v_dev = dev_bits(k_host, dt), dev_bits(v_host, dt)
    bm = BlockManager(NB)
    prompts = {1: 250, 2: 37, 3: 130}
    done = {sid: 0 for sid in prompts}
    for sid in prompts:
        bm.add_sequence(sid)
    # chunked prefill: every step takes up to CHUNK tokens of each unfinished
    # prompt, the chunks of all sequences packed into one call
    while any(done[s] < prompts[s] for s in prompts):
        sids = [s for s in prompts if done[s] < prompts[s]]
        chunks = [min(CHUNK, prompts[s] - done[s]) for s in sids]
        slots = np.concatenate([bm.append(s, c)[0] for s, c in zip(sids, chunks)])
        kn, vn = bits(len(slots), HKV, D), bits(len(slots), HKV, D)
        pa.reshape_and_cache(dev_bits(kn, dt), dev_bits(vn, dt), k_dev, v_dev,
                             torch.from_numpy(slots).cuda())
        oracle.reshape_and_cache(k_host, v_host, kn, vn, slots)
        for s, c in zip(sids, chunks):
            done[s] += c
        tables = np.stack([bm.block_table(s, MAXB)[0] for s in sids])
        lens = np.array([done[s] for s in sids], np.int32)
        qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
        q = bits(int(qs[-1]), HQ, D)
        out = torch.empty(int(qs[-1]), HQ, D, dtype=TORCH_DTYPE[dt], device="cuda")
        pa.prefill(out, dev_bits(q, dt), k_dev, v_dev, torch.from_numpy(tables).cuda(),
                   torch.from_numpy(lens).cuda(), torch.from_numpy(qs).cuda(), max(chunks), scale)
        ref = oracle.prefill(q, k_host, v_host, tables, lens, qs, scale, dt)
        assert max_err(out, ref) <= TOL[dt]
        assert pa.get_device_error() == 0
    # parallel sampling from prompt 1 (250 tokens: its last block is shared
    # and partly filled, so the first token of each sample copies it)
    samples = [1] + [10 + c for c in range(3)]
    for c in samples[1:]:
        bm.fork(1, c)
    live = samples + [2, 3]
    for step in range(5):
        slots = np.empty(len(live), np.int64)
        pairs = []
        for i, sid in enumerate(live):
            sl, cow = bm.append(sid, 1)
            slots[i] = sl[0]
            if cow is not None:
                pairs.append(cow)
        if step == 0:
            assert len(pairs) == len(samples) - 1
        if pairs:
            bmap = np.array(pairs, np.int64)
            pa.copy_blocks(k_dev, v_dev, torch.from_numpy(bmap).cuda())
            oracle.copy_blocks(k_host, v_host, bmap)
        tables = np.stack([bm.block_table(s, MAXB)[0] for s in live])
        lens = np.array([bm.block_table(s, MAXB)[2] for s in live], np.int32)
        q, kn, vn = bits(len(live), HQ, D), bits(len(live), HKV, D), bits(len(live), HKV, D)
        out = torch.empty(len(live), HQ, D, dtype=TORCH_DTYPE[dt], device="cuda")
        pa.decode_append(out, dev_bits(q, dt), k_dev, v_dev, torch.from_numpy(tables).cuda(),
                         torch.from_numpy(lens).cuda(), dev_bits(kn, dt), dev_bits(vn, dt),
                         torch.from_numpy(slots).cuda(), scale)
        oracle.reshape_and_cache(k_host, v_host, kn, vn, slots)
        ref = oracle.decode(q, k_host, v_host, tables, lens, scale, dt)
        assert max_err(out, ref) <= TOL[dt], f"step {step}"
        assert pa.get_device_error() == 0
    assert np.array_equal(host_bits(k_dev), k_host) and np.array_equal(host_bits(v_dev), v_host)
    for sid in live:
        bm.free(sid)
    st = bm.stats()
    assert st["free_blocks"] == NB and st["allocations"] == st["releases"]
