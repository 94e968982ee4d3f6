"""Full-size parity: every synthetic workload at its stated size, one whole
decode step (copy-on-write, reshape_and_cache, decode) in the split mode the
benchmark uses and in the other modes, against the fp64 oracle.  Outputs are
compared element by element; the pools after the step bit-exactly.  Slots
holding no live token are NaN."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, DevWorkload, host_bits, max_err

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# split mode used by the benchmark for each workload, then the others
MODES = {"tiny": (0, -1), "mha7b": (0, -1, 512), "gqa8b": (0, 512, -1), "long": (512, 0),
         "parsamp": (0, 512)}

_cache = {}


def reference(name):
    if name not in _cache:
        _cache.clear()
        w = synth.by_name(name, poison=True)
        _cache[name] = (w, oracle.step(w))
    return _cache[name]


@pytest.mark.parametrize("name", list(MODES))
def test_full_size_step(pa, name):
    w, (ref, k_ref, v_ref) = reference(name)
    for i, mode in enumerate(MODES[name]):
        dw = DevWorkload(w)
        dw.step(pa, partition_size=mode)
        err = max_err(dw.out, ref)
        assert err <= TOL[w.dtype], f"{name} mode {mode}: max|err| {err}"
        assert pa.get_device_error() == 0
        if i == 0:
            assert np.array_equal(host_bits(dw.k), k_ref)
            assert np.array_equal(host_bits(dw.v), v_ref)
        del dw
        torch.cuda.empty_cache()
    if w.slot_mapping is not None:
        # the launch configuration the benchmark times: the append fused into the decode
        dw = DevWorkload(w)
        if dw.pairs is not None:
            pa.copy_blocks(dw.k, dw.v, dw.pairs)
        pa.decode_append(dw.out, dw.q, dw.k, dw.v, dw.tables, dw.lens, dw.k_new, dw.v_new,
                         dw.slots, w.scale, partition_size=MODES[name][0])
        err = max_err(dw.out, ref)
        assert err <= TOL[w.dtype], f"{name} fused append: max|err| {err}"
        assert pa.get_device_error() == 0
        assert np.array_equal(host_bits(dw.k), k_ref)
        assert np.array_equal(host_bits(dw.v), v_ref)
