"""ctypes binding of the host block manager (include/pa_block_manager.h).

A thin wrapper: every operation is the library's C++ code; this module only
converts arguments and results.
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from . import PagedAttnError, load

PA_ERR_OUT_OF_BLOCKS = 6


class BMStats(C.Structure):
    _fields_ = [("num_blocks", C.c_int64), ("free_blocks", C.c_int64),
                ("num_sequences", C.c_int64), ("allocations", C.c_int64),
                ("releases", C.c_int64), ("cow_copies", C.c_int64),
                ("shared_blocks", C.c_int64)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


def _lib():
    L = load()
    if not getattr(L, "_bm_ready", False):
        vp, i, i64 = C.c_void_p, C.c_int, C.c_int64
        L.pa_bm_create.restype = vp
        L.pa_bm_create.argtypes = [i, i]
        L.pa_bm_destroy.restype = None
        L.pa_bm_destroy.argtypes = [vp]
        L.pa_bm_add_sequence.restype = i
        L.pa_bm_add_sequence.argtypes = [vp, i64]
        L.pa_bm_fork.restype = i
        L.pa_bm_fork.argtypes = [vp, i64, i64]
        L.pa_bm_append.restype = i
        L.pa_bm_append.argtypes = [vp, i64, i, vp, vp, C.POINTER(C.c_int)]
        L.pa_bm_free_sequence.restype = i
        L.pa_bm_free_sequence.argtypes = [vp, i64]
        L.pa_bm_block_table.restype = i
        L.pa_bm_block_table.argtypes = [vp, i64, vp, i, C.POINTER(C.c_int),
                                        C.POINTER(C.c_int64)]
        L.pa_bm_ref_count.restype = i
        L.pa_bm_ref_count.argtypes = [vp, i]
        L.pa_bm_get_stats.restype = i
        L.pa_bm_get_stats.argtypes = [vp, C.POINTER(BMStats)]
        L._bm_ready = True
    return L


def _check(fn, rc):
    if rc != 0:
        raise PagedAttnError(fn, rc)


class BlockManager:
    """Free list, reference counts, on-demand allocation and copy-on-write."""

    def __init__(self, num_blocks: int, block_size: int = 16):
        self._L = _lib()
        self._h = self._L.pa_bm_create(num_blocks, block_size)
        if not self._h:
            raise ValueError("bad pool size")
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self):
        if self._h:
            self._L.pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_sequence(self, seq_id: int):
        _check("pa_bm_add_sequence", self._L.pa_bm_add_sequence(self._h, seq_id))

    def fork(self, parent: int, child: int):
        _check("pa_bm_fork", self._L.pa_bm_fork(self._h, parent, child))

    def append(self, seq_id: int, num_tokens: int = 1):
        """(slots int64[num_tokens], cow pair (src, dst) or None)."""
        slots = np.empty(max(1, num_tokens), dtype=np.int64)
        pair = np.empty(2, dtype=np.int64)
        ncow = C.c_int(0)
        _check("pa_bm_append", self._L.pa_bm_append(
            self._h, seq_id, num_tokens, slots.ctypes.data, pair.ctypes.data, C.byref(ncow)))
        return slots[:num_tokens], (tuple(int(x) for x in pair) if ncow.value else None)

    def free(self, seq_id: int):
        _check("pa_bm_free_sequence", self._L.pa_bm_free_sequence(self._h, seq_id))

    def block_table(self, seq_id: int, max_blocks: int):
        """(table int32[max_blocks] padded with -1, number of blocks, sequence length)."""
        t = np.empty(max_blocks, dtype=np.int32)
        nb = C.c_int(0)
        ln = C.c_int64(0)
        _check("pa_bm_block_table", self._L.pa_bm_block_table(
            self._h, seq_id, t.ctypes.data, max_blocks, C.byref(nb), C.byref(ln)))
        return t, nb.value, ln.value

    def ref_count(self, block: int) -> int:
        return self._L.pa_bm_ref_count(self._h, block)

    def stats(self) -> dict:
        st = BMStats()
        _check("pa_bm_get_stats", self._L.pa_bm_get_stats(self._h, C.byref(st)))
        return st.as_dict()
