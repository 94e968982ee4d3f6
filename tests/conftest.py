import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity cases")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(scope="session")
def pa():
    """The CUDA library's binding, built in-tree first (no fallback if that fails)."""
    from paged_kv_cache_260_gb300 import _build
    _build.build()
    import paged_kv_cache_260_gb300 as m
    m.load()
    return m


@pytest.fixture(autouse=True)
def _device_errors_clear(request):
    """GPU tests start with the library's device error bits cleared."""
    if "gpu" in request.keywords:
        import torch
        if torch.cuda.is_available():
            import paged_kv_cache_260_gb300 as m
            if m._lib is not None:
                m.get_device_error(clear=True)
    yield
