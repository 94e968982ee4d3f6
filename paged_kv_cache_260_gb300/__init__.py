"""GB300 (sm_103a) paged KV cache: decode attention, chunked prefill,
reshape_and_cache, copy_blocks, swap_blocks.

A thin ctypes binding over ``libpagedattn.so`` (the C ABI in
``include/pagedattn.h``).  Functions take torch CUDA tensors, pass their data
pointers, sizes and the current stream to the library and raise
``PagedAttnError`` on a non-zero status.  No computation happens here: every
step runs in the library's kernels, and there is no fallback when the library
is missing -- loading it fails loudly.

Names follow the C ABI without the ``pa_`` prefix.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

__all__ = [
    "PagedAttnError", "load", "version", "decode", "decode_workspace_size", "workspace_for",
    "decode_noalloc", "decode_append", "decode_shared_prefix",
    "decode_shared_prefix_workspace_size", "prefill", "prefill_workspace_size",
    "reshape_and_cache", "copy_blocks", "swap_blocks", "gather_kv", "validate_tables",
    "selftest_bounded_wait", "get_device_error",
    "PA_DTYPE_F16", "PA_DTYPE_BF16", "DEVERR", "STATUS",
]

PA_DTYPE_F16 = 0
PA_DTYPE_BF16 = 1
BLOCK_SIZE = 16
STATUS = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_WORKSPACE",
          4: "PA_ERR_CUDA", 5: "PA_ERR_DEVICE"}
DEVERR = {"SLOT_RANGE": 0x1, "BLOCK_RANGE": 0x2, "TABLE_RANGE": 0x4, "SEQLEN_RANGE": 0x8,
          "TIMEOUT": 0x10, "APPEND_SLOT": 0x20, "QUERY_RANGE": 0x40}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedattn.so")
_lib = None
_lock = threading.Lock()


class PagedAttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        name = STATUS.get(status, str(status))
        super().__init__(f"{fn} failed: {name}")


def load(path: str = LIB_PATH):
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    L = _lib
    if L is not None:                    # every call after the first
        return L
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(path)
        vp, i, f, sz = C.c_void_p, C.c_int, C.c_float, C.c_size_t
        L.pa_version.restype = i
        L.pa_version.argtypes = []
        L.pa_status_string.restype = C.c_char_p
        L.pa_status_string.argtypes = [i]
        L.pa_decode_workspace_size.restype = sz
        L.pa_decode_workspace_size.argtypes = [i, i, i, i, i, i]
        L.pa_decode.restype = i
        L.pa_decode.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, vp, sz, vp]
        L.pa_decode_append.restype = i
        L.pa_decode_append.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i,
                                       f, i, i, vp, sz, vp]
        L.pa_decode_shared_prefix_workspace_size.restype = sz
        L.pa_decode_shared_prefix_workspace_size.argtypes = [i, i, i, i, i, i, i]
        L.pa_decode_shared_prefix.restype = i
        L.pa_decode_shared_prefix.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i,
                                              i, i, i, i, f, i, vp, sz, vp]
        L.pa_decode_noalloc.restype = i
        L.pa_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
        L.pa_reshape_and_cache.restype = i
        L.pa_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
        L.pa_copy_blocks.restype = i
        L.pa_copy_blocks.argtypes = [vp, vp, vp, i, i, i, i, i, i, vp]
        L.pa_swap_blocks.restype = i
        L.pa_swap_blocks.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp]
        L.pa_gather_kv.restype = i
        L.pa_gather_kv.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp]
        L.pa_validate_tables.restype = i
        L.pa_validate_tables.argtypes = [vp, vp, i, i, i, i, vp, vp]
        L.pa_prefill.restype = i
        L.pa_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp,
                                 sz, vp]
        L.pa_prefill_workspace_size.restype = sz
        L.pa_prefill_workspace_size.argtypes = [i, i, i, i]
        L.pa_selftest_bounded_wait.restype = i
        L.pa_selftest_bounded_wait.argtypes = [i, vp]
        L.pa_get_device_error.restype = i
        L.pa_get_device_error.argtypes = [vp, C.POINTER(C.c_uint32), i]
        _lib = L
        return L


def version() -> int:
    return load().pa_version()


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float16:
        return PA_DTYPE_F16
    if t.dtype == torch.bfloat16:
        return PA_DTYPE_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    # a plain int: the argtypes (c_void_p) convert it
    return None if t is None else t.data_ptr()


_current_raw_stream = None


def _stream(stream):
    """The stream's handle; by default the current device's current stream,
    read as a raw handle (building a torch.cuda.Stream object for it costs a
    few microseconds a call)."""
    global _current_raw_stream
    if stream is not None:
        return stream.cuda_stream
    if _current_raw_stream is None:
        torch = _torch()
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        dev = getattr(torch._C, "_cuda_getDevice", None)
        if raw is not None and dev is not None:
            torch.cuda.init()
            _current_raw_stream = lambda: raw(dev())
        else:
            _current_raw_stream = lambda: torch.cuda.current_stream().cuda_stream
    return _current_raw_stream()


def _scratch(nbytes, device, stream):
    """A uint8 scratch tensor for one call.  It is tied to the call's stream,
    so the caching allocator does not hand its memory out again before the
    kernels that use it have run."""
    torch = _torch()
    t = torch.empty(nbytes, dtype=torch.uint8, device=device)
    if stream is not None:
        t.record_stream(stream)
    return t


def _check(fn: str, rc: int):
    if rc != 0:
        raise PagedAttnError(fn, rc)


def _require(cond: bool, what: str):
    if not cond:
        raise ValueError(what)


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------
def decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                          partition_size=0) -> int:
    return int(load().pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                               max_blocks_per_seq, partition_size))


def workspace_for(q, k_cache, block_tables, partition_size=0, stream=None):
    """A workspace tensor sized for pa_decode on these shapes (None when none is needed)."""
    n, hq, d = q.shape
    nbytes = decode_workspace_size(n, hq, k_cache.shape[1], d, block_tables.shape[1],
                                   partition_size)
    if nbytes == 0:
        return None
    return _scratch(nbytes, q.device, stream)


def decode(out, q, k_cache, v_cache, block_tables, seq_lens, scale, partition_size=0,
           workspace=None, stream=None):
    """pa_decode: out[s, h] = softmax(scale * q[s, h] . K_s) V_s over the paged pool.

    q, out [num_seqs, num_heads, head_dim]; k_cache, v_cache
    [num_blocks, num_kv_heads, 16, head_dim]; block_tables int32
    [num_seqs, max_blocks]; seq_lens int32 [num_seqs].
    """
    n, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    _require(out.shape == q.shape and d2 == d and v_cache.shape == k_cache.shape, "shapes")
    _require(block_tables.dim() == 2 and block_tables.shape[0] == n and seq_lens.shape == (n,),
             "table shapes")
    for t in (out, q, k_cache, v_cache, block_tables, seq_lens):
        _require(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")
    if workspace is None:
        workspace = workspace_for(q, k_cache, block_tables, partition_size, stream)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().pa_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                          _ptr(seq_lens), n, hq, hkv, d, bs, block_tables.shape[1], nb,
                          float(scale), _dtype_code(q), int(partition_size), _ptr(workspace),
                          wbytes, _stream(stream))
    _check("pa_decode", rc)
    return out


def decode_append(out, q, k_cache, v_cache, block_tables, seq_lens, k_new, v_new, slot_mapping,
                  scale, partition_size=0, workspace=None, stream=None):
    """pa_decode_append: reshape_and_cache of each sequence's newest token, then decode,
    in one launch.  slot_mapping[s] is the slot of position seq_lens[s] - 1 (or < 0)."""
    n, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    _require(out.shape == q.shape and d2 == d and v_cache.shape == k_cache.shape, "shapes")
    _require(block_tables.dim() == 2 and block_tables.shape[0] == n and seq_lens.shape == (n,),
             "table shapes")
    _require(k_new.shape == (n, hkv, d) and v_new.shape == k_new.shape and
             slot_mapping.shape == (n,), "new-token shapes")
    if workspace is None:
        workspace = workspace_for(q, k_cache, block_tables, partition_size, stream)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().pa_decode_append(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(block_tables), _ptr(seq_lens), _ptr(k_new), _ptr(v_new),
                                 _ptr(slot_mapping), n, hq, hkv, d, bs, block_tables.shape[1], nb,
                                 float(scale), _dtype_code(q), int(partition_size),
                                 _ptr(workspace), wbytes, _stream(stream))
    _check("pa_decode_append", rc)
    return out


def decode_shared_prefix_workspace_size(num_seqs, group_size, prefix_len, num_heads,
                                        num_kv_heads, head_dim, max_blocks_per_seq) -> int:
    return int(load().pa_decode_shared_prefix_workspace_size(
        num_seqs, group_size, prefix_len, num_heads, num_kv_heads, head_dim, max_blocks_per_seq))


def decode_shared_prefix(out, q, k_cache, v_cache, block_tables, seq_lens, group_size,
                         prefix_len, scale, k_new=None, v_new=None, slot_mapping=None,
                         workspace=None, stream=None):
    """pa_decode_shared_prefix: decode (with the newest tokens appended when
    k_new, v_new and slot_mapping are given) of a batch whose consecutive
    groups of `group_size` sequences share their first `prefix_len` tokens'
    blocks; the shared prefix is read once per group."""
    n, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    _require(out.shape == q.shape and d2 == d and v_cache.shape == k_cache.shape, "shapes")
    _require(block_tables.dim() == 2 and block_tables.shape[0] == n and seq_lens.shape == (n,),
             "table shapes")
    if k_new is not None:
        _require(k_new.shape == (n, hkv, d) and v_new.shape == k_new.shape and
                 slot_mapping.shape == (n,), "new-token shapes")
    if workspace is None:
        nbytes = decode_shared_prefix_workspace_size(n, group_size, prefix_len, hq, hkv, d,
                                                     block_tables.shape[1])
        workspace = _scratch(nbytes, q.device, stream) if nbytes else None
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().pa_decode_shared_prefix(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(seq_lens),
        _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), n, int(group_size), int(prefix_len), hq,
        hkv, d, bs, block_tables.shape[1], nb, float(scale), _dtype_code(q), _ptr(workspace),
        wbytes, _stream(stream))
    _check("pa_decode_shared_prefix", rc)
    return out


def prefill_workspace_size(num_seqs, max_query_len, num_heads, num_kv_heads) -> int:
    return int(load().pa_prefill_workspace_size(num_seqs, max_query_len, num_heads, num_kv_heads))


def prefill(out, q, k_cache, v_cache, block_tables, seq_lens, query_start, max_query_len, scale,
            workspace="auto", stream=None):
    """pa_prefill: causal attention of each sequence's newest chunk over the paged pool.

    q, out [total_q, num_heads, head_dim], the chunks packed back to back;
    query_start int32 [num_seqs + 1]; seq_lens int32 [num_seqs] counts the
    chunk; max_query_len (host int) is the longest chunk.  workspace: "auto"
    allocates the work-order buffer, None runs without it, or a CUDA uint8
    tensor of at least prefill_workspace_size(...) bytes.
    """
    t, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    n = seq_lens.shape[0]
    _require(out.shape == q.shape and d2 == d and v_cache.shape == k_cache.shape, "shapes")
    _require(block_tables.dim() == 2 and block_tables.shape[0] == n and
             query_start.shape == (n + 1,), "table shapes")
    for x in (out, q, k_cache, v_cache, block_tables, seq_lens, query_start):
        _require(x.is_cuda and x.is_contiguous(), "tensors must be contiguous CUDA tensors")
    if isinstance(workspace, str):
        nbytes = prefill_workspace_size(n, int(max_query_len), hq, hkv)
        workspace = _scratch(nbytes, q.device, stream) if nbytes else None
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().pa_prefill(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                           _ptr(seq_lens), _ptr(query_start), n, int(max_query_len), hq, hkv, d,
                           bs, block_tables.shape[1], nb, float(scale), _dtype_code(q),
                           _ptr(workspace), wbytes, _stream(stream))
    _check("pa_prefill", rc)
    return out


def decode_noalloc(out, q, k_cache, v_cache, block_tables, seq_lens, scale, stream=None):
    """pa_decode_noalloc: decode with the library's own fixed scratch (balanced split).

    For callers that cannot allocate a workspace.  Calls share one scratch
    array per device, so calls that may overlap on the GPU must be ordered on
    one stream; the first call on a device must come before any stream capture.
    """
    n, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    _require(out.shape == q.shape and d2 == d and v_cache.shape == k_cache.shape, "shapes")
    _require(block_tables.dim() == 2 and block_tables.shape[0] == n and seq_lens.shape == (n,),
             "table shapes")
    rc = load().pa_decode_noalloc(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(block_tables), _ptr(seq_lens), n, hq, hkv, d, bs,
                                  block_tables.shape[1], nb, float(scale), _dtype_code(q),
                                  _stream(stream))
    _check("pa_decode_noalloc", rc)
    return out


def reshape_and_cache(k_new, v_new, k_cache, v_cache, slot_mapping, stream=None):
    """pa_reshape_and_cache: write token i's K/V into pool slot slot_mapping[i] (<0 skips)."""
    nt, hkv, d = k_new.shape
    nb, hkv2, bs, d2 = k_cache.shape
    _require(hkv == hkv2 and d == d2 and v_new.shape == k_new.shape, "shapes")
    _require(slot_mapping.shape == (nt,), "slot_mapping shape")
    rc = load().pa_reshape_and_cache(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(slot_mapping), nt, hkv, d, bs, nb, _dtype_code(k_cache),
                                     _stream(stream))
    _check("pa_reshape_and_cache", rc)


def copy_blocks(k_cache, v_cache, block_mapping, stream=None):
    """pa_copy_blocks: whole-block copies src -> dst for each row of block_mapping [P, 2]."""
    nb, hkv, bs, d = k_cache.shape
    _require(block_mapping.dim() == 2 and block_mapping.shape[1] == 2, "block_mapping shape")
    rc = load().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(block_mapping),
                               block_mapping.shape[0], hkv, d, bs, nb, _dtype_code(k_cache),
                               _stream(stream))
    _check("pa_copy_blocks", rc)


def swap_blocks(dst_k, dst_v, src_k, src_v, block_mapping, stream=None):
    """pa_swap_blocks: whole-block copies src -> dst between two pools (one of them
    typically in page-locked host memory, e.g. ``torch.empty(..).pin_memory()``)."""
    snb, hkv, bs, d = src_k.shape
    dnb = dst_k.shape[0]
    _require(dst_k.shape[1:] == src_k.shape[1:] and dst_v.shape == dst_k.shape and
             src_v.shape == src_k.shape, "pool shapes")
    _require(block_mapping.dim() == 2 and block_mapping.shape[1] == 2, "block_mapping shape")
    rc = load().pa_swap_blocks(_ptr(dst_k), _ptr(dst_v), _ptr(src_k), _ptr(src_v),
                               _ptr(block_mapping), block_mapping.shape[0], hkv, d, bs, snb, dnb,
                               _dtype_code(src_k), _stream(stream))
    _check("pa_swap_blocks", rc)


def gather_kv(k_out, v_out, k_cache, v_cache, block_tables, seq_lens, stream=None):
    """pa_gather_kv: k_out[s, h, t] = k_cache[table[s][t//16], h, t%16] for t < seq_lens[s]."""
    nb, hkv, bs, d = k_cache.shape
    n, mb = block_tables.shape
    _require(k_out.shape == (n, hkv, mb * bs, d) and v_out.shape == k_out.shape, "out shape")
    rc = load().pa_gather_kv(_ptr(k_out), _ptr(v_out), _ptr(k_cache), _ptr(v_cache),
                             _ptr(block_tables), _ptr(seq_lens), n, hkv, d, bs, mb, nb,
                             _dtype_code(k_cache), _stream(stream))
    _check("pa_gather_kv", rc)


def validate_tables(block_tables, seq_lens, num_blocks, bad_count, stream=None):
    """pa_validate_tables: adds to bad_count (uint32/int32 device scalar) the bad entries."""
    n, mb = block_tables.shape
    rc = load().pa_validate_tables(_ptr(block_tables), _ptr(seq_lens), n, mb, num_blocks,
                                   BLOCK_SIZE, _ptr(bad_count), _stream(stream))
    _check("pa_validate_tables", rc)


def selftest_bounded_wait(limit_us=2000, stream=None):
    """pa_selftest_bounded_wait: a copy wait that must time out and report it."""
    _check("pa_selftest_bounded_wait", load().pa_selftest_bounded_wait(int(limit_us),
                                                                       _stream(stream)))


def get_device_error(clear=True, stream=None) -> int:
    """Synchronise and return (and by default clear) the PA_DEVERR_* bits."""
    bits = C.c_uint32(0)
    rc = load().pa_get_device_error(_stream(stream), C.byref(bits), 1 if clear else 0)
    if rc not in (0, 5):
        _check("pa_get_device_error", rc)
    return int(bits.value)
