"""pa_decode_noalloc: the decode entry point that allocates nothing.

For callers that cannot allocate device memory (an engine that gave its free
HBM to the KV block pool, a plugin handed only inputs and outputs), the
library keeps the split-K scratch in a fixed device array of its own.  This
checks, through the C ABI, that two calls in a row on different workloads --
the second reusing the scratch the first left behind -- match pa_decode,
which takes a caller-owned workspace, within the decode tolerance, and that
sizes beyond the array are refused.  This file is collected last.
"""
import pytest
import torch

import synth
from gpu_util import TOL, DevWorkload, to_f64

pytestmark = pytest.mark.gpu


def _compare(pa, w):
    dw = DevWorkload(w)
    pa.reshape_and_cache(dw.k_new, dw.v_new, dw.k, dw.v, dw.slots)
    ref = torch.empty_like(dw.q)
    pa.decode(ref, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale, partition_size=0)
    got = torch.full_like(dw.q, float("nan"))
    pa.decode_noalloc(got, dw.q, dw.k, dw.v, dw.tables, dw.lens, w.scale)
    torch.cuda.synchronize()
    err = float((to_f64(got) - to_f64(ref)).__abs__().max())
    assert err <= TOL[w.dtype], f"max|err| {err}"
    assert pa.get_device_error() == 0


def test_noalloc_matches_decode_twice(pa):
    _compare(pa, synth.gqa8b(poison=True))                       # bf16, group 4, 128 seqs
    _compare(pa, synth.build("second", 40, 40, 8, 64, "f16",     # f16, group 5, other sizes
                             list(range(1, 2000, 50)), seed=77, append=True, poison=True))


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
