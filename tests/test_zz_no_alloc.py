"""pa_decode_noalloc: the decode entry point that allocates nothing.

Some callers cannot allocate device memory at all: an engine that gave its
free HBM to the KV block pool at start-up, a plugin whose host framework
hands it only inputs and outputs, code where cudaMalloc is not allowed.  For
them the library keeps the split-K scratch in a fixed device array of its
own.  Through the C ABI, two calls in a row on different workloads (the
second reusing whatever the first left in the shared scratch) must match the
fp64 oracle within the decode tolerance, and match pa_decode with a
caller-owned workspace bit for bit (same kernels, same split).  Sizes beyond
the array are refused before anything is launched.  This file is collected
last, so a run that stops at the first failure has run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, DevWorkload, max_err

pytestmark = pytest.mark.gpu


def _check(pa, w):
    dw = DevWorkload(w)
    if dw.pairs is not None:
        pa.copy_blocks(dw.k, dw.v, dw.pairs)
    if dw.slots is not None:
        pa.reshape_and_cache(dw.k_new, dw.v_new, dw.k, dw.v, dw.slots)
    got = torch.full_like(dw.q, float("nan"))
    pa.decode_noalloc(got, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale)
    ref_gpu = torch.full_like(dw.q, float("nan"))
    pa.decode(ref_gpu, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale, partition_size=0)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    ref, _, _ = oracle.step(w)
    err = max_err(got, ref)                       # also fails on any NaN left in `got`
    assert err <= TOL[w.dtype], f"{w.name}: max|err| {err} vs the oracle"
    assert torch.equal(got.view(torch.int16), ref_gpu.view(torch.int16)), \
        f"{w.name}: differs from pa_decode with a caller-owned workspace"


def test_noalloc_matches_oracle_twice(pa):
    # bf16, group 4, 128 ragged sequences, NaN in every slot no live token holds
    _check(pa, synth.gqa8b(poison=True))
    # then f16, group 5, head_dim 64, lengths 1..1951 cut across workers, on
    # the scratch the first call left behind
    _check(pa, synth.build("second", 40, 40, 8, 64, "f16", list(range(1, 2000, 50)), seed=77,
                           append=True, poison=True))


def test_noalloc_empty_batch_checks_arguments(pa):
    q = torch.zeros(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    tables = torch.zeros(0, 1, dtype=torch.int32, device="cuda")
    lens = torch.zeros(0, dtype=torch.int32, device="cuda")
    pa.decode_noalloc(q, q, k, k, tables, lens, 0.1)             # nothing to do: ok
    L = pa.load()
    s = torch.cuda.current_stream().cuda_stream
    for bad_hd in (96,):                                          # unsupported head_dim
        a = [q.data_ptr(), q.data_ptr(), k.data_ptr(), k.data_ptr(), tables.data_ptr(),
             lens.data_ptr(), 0, 8, 2, bad_hd, 16, 1, 4]
        rc_dec = L.pa_decode(*a, 0.1, 1, 0, None, 0, s)
        rc_na = L.pa_decode_noalloc(*a, 0.1, 1, s)
        assert rc_dec == rc_na == 2                               # PA_ERR_UNSUPPORTED


def test_noalloc_refuses_sizes_beyond_its_scratch(pa):
    limit = 16 << 20                                  # PA_NOALLOC_SCRATCH_BYTES
    # group 8 at head_dim 128 needs the most scratch per thread block
    n, hq, hkv, d = 64, 64, 8, 128
    need = pa.decode_workspace_size(n, hq, hkv, d, 1, 0)
    if need <= limit:
        pytest.skip(f"this GPU needs only {need} bytes of scratch for the largest group")
    q = torch.zeros(n, hq, d, dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(q, 7.0)
    k = torch.zeros(1, hkv, 16, d, dtype=torch.bfloat16, device="cuda")
    tables = torch.zeros(n, 1, dtype=torch.int32, device="cuda")
    lens = torch.ones(n, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PagedAttnError) as e:
        pa.decode_noalloc(out, q, k, k, tables, lens, 0.1)
    assert e.value.status == 3                        # PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())                   # nothing was launched
