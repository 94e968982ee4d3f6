"""Decode steps driven by the host block manager: prompts are written, forked
into samples, and every step appends one token per sample.  The manager's
copy-on-write pairs go to copy_blocks and its slots to decode_append.  Each
step is checked against the oracle run on a host replica of the pool; at the
end the pools are bit-identical and freeing every sequence leaks nothing."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, dev_bits, host_bits, max_err
from paged_kv_cache_260_gb300.block_manager import BlockManager

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("prompt_lens,mode", [((40, 37), 0), ((32, 50), -1), ((40, 37), 16)])
def test_parallel_sampling_steps_with_the_block_manager(pa, prompt_lens, mode):
    rng = np.random.default_rng(7)
    NB, HKV, HQ, D, S, STEPS, MAXB = 96, 2, 8, 128, 4, 6, 8
    dt = "f16"

    def bits(*shape):
        return synth.to_bits(rng.standard_normal(shape).astype(np.float32), dt)

    k_host = bits(NB, HKV, 16, D)                            # stale contents everywhere
    v_host = bits(NB, HKV, 16, D)
    k_dev, v_dev = dev_bits(k_host, dt), dev_bits(v_host, dt)
    bm = BlockManager(NB)
    samples = []
    for p, L in enumerate(prompt_lens):
        root = 1000 * p
        bm.add_sequence(root)
        slots, cow = bm.append(root, L)
        assert cow is None
        kn, vn = bits(L, HKV, D), bits(L, HKV, D)
        pa.reshape_and_cache(dev_bits(kn, dt), dev_bits(vn, dt), k_dev, v_dev,
                             torch.from_numpy(slots).cuda())
        oracle.reshape_and_cache(k_host, v_host, kn, vn, slots)
        samples.append(root)
        for c in range(1, S):
            bm.fork(root, root + c)
            samples.append(root + c)
    n = len(samples)
    for step in range(STEPS):
        slots = np.empty(n, np.int64)
        pairs = []
        for i, sid in enumerate(samples):
            sl, cow = bm.append(sid, 1)
            slots[i] = sl[0]
            if cow is not None:
                pairs.append(cow)
        tables = np.stack([bm.block_table(sid, MAXB)[0] for sid in samples])
        lens = np.array([bm.block_table(sid, MAXB)[2] for sid in samples], np.int32)
        q, kn, vn = bits(n, HQ, D), bits(n, HKV, D), bits(n, HKV, D)
        if pairs:
            bmap = np.array(pairs, np.int64)
            pa.copy_blocks(k_dev, v_dev, torch.from_numpy(bmap).cuda())
            oracle.copy_blocks(k_host, v_host, bmap)
        out = torch.empty(n, HQ, D, dtype=torch.float16, device="cuda")
        pa.decode_append(out, dev_bits(q, dt), k_dev, v_dev, torch.from_numpy(tables).cuda(),
                         torch.from_numpy(lens).cuda(), dev_bits(kn, dt), dev_bits(vn, dt),
                         torch.from_numpy(slots).cuda(), 1 / np.sqrt(D), partition_size=mode)
        oracle.reshape_and_cache(k_host, v_host, kn, vn, slots)
        ref = oracle.decode(q, k_host, v_host, tables, lens, 1 / np.sqrt(D), dt)
        assert max_err(out, ref) <= TOL[dt], f"step {step}"
        assert pa.get_device_error() == 0
        if step == 0:
            # first token after an unaligned prompt: every sample but the last to
            # write copies the shared partial block
            unaligned = sum(1 for L in prompt_lens if L % 16)
            assert len(pairs) == unaligned * (S - 1)
    assert np.array_equal(host_bits(k_dev), k_host) and np.array_equal(host_bits(v_dev), v_host)
    for sid in samples:
        bm.free(sid)
    st = bm.stats()
    assert st["free_blocks"] == NB and st["allocations"] == st["releases"]
