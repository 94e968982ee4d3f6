"""The C-ABI library builds, loads and exports every entry point its header
declares; host-side argument checks return their status codes without
touching a GPU (all these calls fail validation before any CUDA call)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_260_gb300 import _build
    import paged_kv_cache_260_gb300 as pa
    _build.build()
    return pa.load()


def declared_symbols():
    syms = set()
    inc = os.path.join(ROOT, "include")
    for name in os.listdir(inc):
        if name.endswith(".h"):
            text = open(os.path.join(inc, name)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            syms |= set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text))
    return syms


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("pa_decode", "pa_prefill", "pa_reshape_and_cache", "pa_copy_blocks",
              "pa_decode_workspace_size",
              "pa_gather_kv", "pa_validate_tables", "pa_get_device_error", "pa_status_string",
              "pa_version"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    for s in declared_symbols():
        assert hasattr(lib, s), s


def test_version_and_status_strings(lib):
    assert lib.pa_version() == 1
    assert lib.pa_status_string(0) == b"ok"
    assert lib.pa_status_string(3) == b"workspace missing or too small"


def _decode(lib, **kw):
    a = dict(out=None, q=None, k=None, v=None, tables=None, lens=None, num_seqs=4, num_heads=8,
             num_kv_heads=2, head_dim=128, block_size=16, max_blocks=8, num_blocks=64, scale=0.1,
             dtype=0, partition_size=0, ws=None, ws_bytes=0, stream=None)
    a.update(kw)
    return lib.pa_decode(a["out"], a["q"], a["k"], a["v"], a["tables"], a["lens"], a["num_seqs"],
                         a["num_heads"], a["num_kv_heads"], a["head_dim"], a["block_size"],
                         a["max_blocks"], a["num_blocks"], C.c_float(a["scale"]), a["dtype"],
                         a["partition_size"], a["ws"], a["ws_bytes"], a["stream"])


def test_decode_rejects_bad_scalars(lib):
    assert _decode(lib, head_dim=96) == 2              # PA_ERR_UNSUPPORTED
    assert _decode(lib, block_size=32) == 2
    assert _decode(lib, dtype=7) == 2
    assert _decode(lib, num_heads=7) == 1              # not a multiple of kv heads
    assert _decode(lib, num_heads=34) == 2             # group 17 > 16
    assert _decode(lib, num_heads=32) == 1             # group 16 is served: null pointers refused
    assert _decode(lib, scale=float("nan")) == 1
    assert _decode(lib, num_seqs=-1) == 1
    assert _decode(lib, num_seqs=0) == 0               # nothing to do
    assert _decode(lib) == 1                           # null pointers
    fake = C.c_void_p(0x1000)
    assert _decode(lib, out=fake, q=C.c_void_p(0x1008), k=fake, v=fake, tables=fake,
                   lens=fake) == 1                     # misaligned q


def test_decode_append_requires_the_new_tokens(lib):
    fake = C.c_void_p(0x1000)
    args = [fake] * 6 + [None, None, None, 4, 8, 2, 128, 16, 8, 64, C.c_float(0.1), 0, 0, None,
                         0, None]
    assert lib.pa_decode_append(*args) == 1          # k_new, v_new, slot_mapping missing
    args[6:9] = [fake, C.c_void_p(0x1008), fake]
    assert lib.pa_decode_append(*args) == 1          # misaligned v_new


def test_cache_entry_points_reject_bad_scalars(lib):
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 4, 8, 96, 16, 64, 0, None) == 2
    assert lib.pa_reshape_and_cache(None, None, None, None, None, -1, 8, 64, 16, 64, 0, None) == 1
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 0, 8, 64, 16, 64, 0, None) == 0
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 4, 8, 64, 16, 64, 0, None) == 1
    assert lib.pa_copy_blocks(None, None, None, 3, 8, 128, 8, 64, 0, None) == 2
    assert lib.pa_copy_blocks(None, None, None, 3, 8, 128, 16, 64, 0, None) == 1
    assert lib.pa_copy_blocks(None, None, None, 0, 8, 128, 16, 64, 1, None) == 0
    assert lib.pa_gather_kv(None, None, None, None, None, None, 2, 8, 128, 16, 4, 64, 0, None) == 1
    assert lib.pa_validate_tables(None, None, 2, 4, 64, 16, None, None) == 1
    assert lib.pa_validate_tables(None, None, 2, 4, 64, 8, None, None) == 2


def test_fixed_partition_workspace_size(lib):
    # documented part: m and l S*Hq*P floats each, o S*Hq*P*D floats, each array
    # 256-byte aligned; per-worker slots follow, sized by the device's SM count
    S, Hq, Hkv, D, mb, P = 4, 32, 8, 128, 8192, 512
    pmax = (mb * 16 + P - 1) // P
    rows = S * Hq * pmax

    def up(x):
        return (x + 255) // 256 * 256

    documented = up(up(up(4 * rows) + 4 * rows) + 4 * rows * D)
    got = lib.pa_decode_workspace_size(S, Hq, Hkv, D, mb, P)
    assert got == 0 or got > documented          # 0: no device to size the slots for
    assert lib.pa_decode_workspace_size(S, Hq, Hkv, D, mb, -1) == 0
    assert lib.pa_decode_workspace_size(S, Hq, Hkv, D, mb, 24) == 0     # not a multiple of 16


def test_prefill_rejects_bad_scalars(lib):
    fake = C.c_void_p(0x1000)

    def call(**kw):
        a = dict(ptrs=[None] * 7, num_seqs=2, max_q=32, hq=8, hkv=2, d=128, bs=16, maxb=8,
                 nb=64, scale=0.1, dtype=1)
        a.update(kw)
        return lib.pa_prefill(*a["ptrs"], a["num_seqs"], a["max_q"], a["hq"], a["hkv"], a["d"],
                              a["bs"], a["maxb"], a["nb"], C.c_float(a["scale"]), a["dtype"],
                              a.get("ws"), a.get("ws_bytes", 0), None)

    assert call(d=96) == 2
    assert call(bs=32) == 2
    assert call(hq=7) == 1
    assert call(hq=258, hkv=1) == 2                  # group over 128 rows
    assert call(scale=float("inf")) == 1
    assert call(scale=-0.1) == 1 and call(scale=0.0) == 1
    assert call(max_q=-1) == 1
    assert call(num_seqs=0) == 0 and call(max_q=0) == 0
    assert call() == 1                               # null pointers
    assert call(ptrs=[fake, C.c_void_p(0x1008)] + [fake] * 5) == 1   # misaligned q
    # a workspace smaller than pa_prefill_workspace_size, or misaligned
    assert call(ptrs=[fake] * 7, ws=fake, ws_bytes=16) == 3
    assert call(ptrs=[fake] * 7, ws=C.c_void_p(0x1010), ws_bytes=4096) == 3


def test_prefill_workspace_size(lib):
    lib.pa_prefill_workspace_size.restype = C.c_size_t
    # 32 q heads over 8 kv heads: 4 per group, 64 chunk tokens per block
    # 16 + 4 * seqs * query tiles + 8 * seqs, rounded up to 256
    assert lib.pa_prefill_workspace_size(8, 512, 32, 8) == 512          # 16 + 256 + 64
    assert lib.pa_prefill_workspace_size(100, 1000, 32, 8) == 7424      # 16 + 6400 + 800
    assert lib.pa_prefill_workspace_size(0, 512, 32, 8) == 0
    assert lib.pa_prefill_workspace_size(8, 512, 30, 8) == 0            # not a multiple
