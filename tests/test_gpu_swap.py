"""GPU parity of pa_swap_blocks: KV blocks moved between the GPU pool and a
pool in page-locked host memory (preemption by swapping), bit-exact against
the oracle, and a decode after swapping back into other blocks unchanged."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import DevWorkload, dev_bits, host_bits

pytestmark = pytest.mark.gpu


def _workload():
    return synth.build("swap", 8, 32, 8, 128, "bf16", [40, 700, 300, 17, 64, 5, 1500, 256],
                       seed=18, pool_factor=3.0, poison=True)


def test_swap_out_and_in_round_trip(pa):
    w = _workload()
    dw = DevWorkload(w)
    pa.decode(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale)
    before = dw.out.clone()
    # preempt sequences 1 and 6: their blocks go to a host pool
    victims = [1, 6]
    blocks = np.concatenate([w.block_tables[s, :synth.cdiv(int(w.seq_lens[s]), 16)] for s in victims])
    nh = len(blocks) + 4
    host_k = torch.zeros((nh,) + tuple(dw.k.shape[1:]), dtype=dw.k.dtype).pin_memory()
    host_v = torch.zeros_like(host_k).pin_memory()
    out_pairs = np.stack([blocks, 2 + np.arange(len(blocks))], 1).astype(np.int64)
    pa.swap_blocks(host_k, host_v, dw.k, dw.v, torch.from_numpy(out_pairs).cuda())
    torch.cuda.synchronize()
    hk = np.zeros((nh,) + w.k_cache.shape[1:], np.uint16)
    hv = np.zeros_like(hk)
    assert oracle.swap_blocks(hk, hv, w.k_cache, w.v_cache, out_pairs) == 0
    assert np.array_equal(host_bits(host_k), hk) and np.array_equal(host_bits(host_v), hv)

    # back into other device blocks, tables remapped: same output, bit for bit
    free = np.setdiff1d(np.arange(w.num_blocks), w.block_tables[w.block_tables >= 0])
    new_ids = np.random.default_rng(4).choice(free, size=len(blocks), replace=False)
    in_pairs = np.stack([2 + np.arange(len(blocks)), new_ids], 1).astype(np.int64)
    pa.swap_blocks(dw.k, dw.v, host_k, host_v, torch.from_numpy(in_pairs).pin_memory())
    tables = w.block_tables.copy()
    i = 0
    for s in victims:
        nb = synth.cdiv(int(w.seq_lens[s]), 16)
        tables[s, :nb] = new_ids[i:i + nb]
        i += nb
    pa.decode(dw.out, dw.q, dw.k, dw.v, torch.from_numpy(tables).cuda(), dw.lens, w.scale)
    assert torch.equal(before, dw.out)
    assert pa.get_device_error() == 0


def test_swap_refuses_pageable_memory(pa):
    w = _workload()
    dw = DevWorkload(w)
    host_k = torch.zeros((4,) + tuple(dw.k.shape[1:]), dtype=dw.k.dtype)   # not page-locked
    host_v = torch.zeros_like(host_k)
    pairs = torch.tensor([[int(w.block_tables[0, 0]), 0]], dtype=torch.int64, device="cuda")
    with pytest.raises(pa.PagedAttnError) as e:
        pa.swap_blocks(host_k, host_v, dw.k, dw.v, pairs)
    assert e.value.status == 1


def test_swap_pairs_outside_a_pool_are_skipped(pa):
    w = _workload()
    dw = DevWorkload(w)
    host_k = torch.zeros((2,) + tuple(dw.k.shape[1:]), dtype=dw.k.dtype).pin_memory()
    host_v = torch.zeros_like(host_k).pin_memory()
    pairs = torch.tensor([[int(w.block_tables[1, 0]), 0], [int(w.block_tables[1, 1]), 5]],
                         dtype=torch.int64, device="cuda")
    pa.swap_blocks(host_k, host_v, dw.k, dw.v, pairs)
    torch.cuda.synchronize()
    assert torch.equal(host_k[0].view(torch.int16), dw.k[int(w.block_tables[1, 0])].view(torch.int16).cpu())
    assert not host_k[1].view(torch.int16).any()
    assert pa.get_device_error() == pa.DEVERR["BLOCK_RANGE"]
