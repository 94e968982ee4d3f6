"""fp64 CPU oracle for paged decode attention, chunked prefill over the same
pool, and the KV-pool kernels.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only users.  The library never imports
this package and this package never imports the library.

The arithmetic lives in ``oracle.c`` (plain C, double precision); this module
compiles it with gcc, loads it with ctypes and runs disjoint ranges of
sequences on threads (ctypes releases the GIL during the call, and each C call
is single-threaded, so threading changes no result).

``brute.py`` next to it is an independent pure-Python restatement for tiny
inputs, used to pin the C code.
"""
from __future__ import annotations

import concurrent.futures as _cf
import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, no fast-math, no FMA contraction)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB)
        L.oracle_decode_bits.argtypes = [_f64p, _u16p, C.c_long, C.c_int]
        L.oracle_decode_bits.restype = None
        L.oracle_attend.argtypes = [_f64p, _f64p, _f64p, _u16p, _u16p, _u16p, _i32p,
                                    C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                    C.c_double, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int]
        L.oracle_attend.restype = None
        L.oracle_decode.argtypes = [_f64p, _u16p, _u16p, _u16p, _i32p, _i32p,
                                    C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                    C.c_double, C.c_int, C.c_int, C.c_int]
        L.oracle_decode.restype = None
        L.oracle_partials.argtypes = [_f64p, _f64p, _f64p, _u16p, _u16p, _u16p, _i32p,
                                      _i32p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                      C.c_double, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int]
        L.oracle_partials.restype = None
        L.oracle_lse_merge.argtypes = [_f64p, _f64p, _f64p, _f64p, C.c_int, C.c_int]
        L.oracle_lse_merge.restype = None
        L.oracle_gather_kv.argtypes = [_u16p, _u16p, _u16p, _u16p, _i32p, C.c_int,
                                       C.c_int, C.c_int, C.c_int, C.c_int, C.c_int]
        L.oracle_gather_kv.restype = None
        L.oracle_reshape_and_cache.argtypes = [_u16p, _u16p, _u16p, _u16p, _i64p,
                                               C.c_int, C.c_int, C.c_int, C.c_int, C.c_long]
        L.oracle_reshape_and_cache.restype = C.c_long
        L.oracle_copy_blocks.argtypes = [_u16p, _u16p, _i64p, C.c_int, C.c_int, C.c_int,
                                         C.c_int, C.c_long]
        L.oracle_copy_blocks.restype = C.c_long
        L.oracle_swap_blocks.argtypes = [_u16p, _u16p, _u16p, _u16p, _i64p, C.c_int, C.c_int,
                                         C.c_int, C.c_int, C.c_long, C.c_long]
        L.oracle_swap_blocks.restype = C.c_long
        L.oracle_prefill.argtypes = [_f64p, _u16p, _u16p, _u16p, _i32p, _i32p, _i32p, C.c_int,
                                     C.c_int, C.c_int, C.c_int, C.c_int, C.c_double, C.c_int,
                                     C.c_int, C.c_int]
        L.oracle_prefill.restype = None
        _lib = L
    return _lib


DTYPES = {"f16": 0, "bf16": 1}
BLOCK_SIZE = 16


def num_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def decode_bits(bits, dtype: str) -> np.ndarray:
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib().oracle_decode_bits(out.reshape(-1), b.reshape(-1), b.size, DTYPES[dtype])
    return out


def _ranges(n, parts):
    parts = max(1, min(parts, n))
    step = (n + parts - 1) // parts
    return [(i, min(n, i + step)) for i in range(0, n, step)]


def decode(q, k_cache, v_cache, block_tables, seq_lens, scale, dtype: str,
           num_kv_heads=None, threads=None, seqs=None) -> np.ndarray:
    """Decode output [num_seqs, Hq, D] in fp64 for every sequence (or ``seqs``)."""
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    block_tables = _c(block_tables, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    S, Hq, D = q.shape
    Hkv = k_cache.shape[1] if num_kv_heads is None else num_kv_heads
    out = np.zeros((S, Hq, D), dtype=np.float64)
    L = lib()
    mb = block_tables.shape[1]
    dt = DTYPES[dtype]

    nt = threads or num_threads()
    sel = list(range(S)) if seqs is None else [int(s) for s in seqs]

    def run(r):
        L.oracle_decode(out, q, k_cache, v_cache, block_tables, seq_lens, Hq, Hkv, D,
                        BLOCK_SIZE, mb, float(scale), dt, r[0], r[1])

    def run_head(sh):
        # one (sequence, head) at a time, for batches too small to spread by sequence
        s, h = sh
        m = np.zeros(1)
        l = np.zeros(1)
        L.oracle_attend(out[s, h], m, l, q, k_cache, v_cache, block_tables, mb, Hq, Hkv, D,
                        BLOCK_SIZE, float(scale), dt, s, h, 0, int(seq_lens[s]))

    if nt > 1 and len(sel) < 2 * nt:
        tasks, fn = [(s, h) for s in sel for h in range(Hq)], run_head
    elif seqs is not None:
        tasks, fn = [(s, s + 1) for s in sel], run
    else:
        tasks, fn = _ranges(S, 4 * nt), run
    if nt == 1 or len(tasks) == 1:
        for t in tasks:
            fn(t)
    else:
        with _cf.ThreadPoolExecutor(nt) as ex:
            list(ex.map(fn, tasks))
    return out


def attend(q, k_cache, v_cache, block_tables, scale, dtype, s, h, t0, t1):
    """(o, m, l) of one head over tokens [t0, t1)."""
    q = _c(q, np.uint16)
    S, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    o = np.zeros(D, dtype=np.float64)
    m = np.zeros(1, dtype=np.float64)
    l = np.zeros(1, dtype=np.float64)
    block_tables = _c(block_tables, np.int32)
    lib().oracle_attend(o, m, l, q, _c(k_cache, np.uint16), _c(v_cache, np.uint16),
                        block_tables, block_tables.shape[1], Hq, Hkv, D, BLOCK_SIZE,
                        float(scale), DTYPES[dtype], s, h, t0, t1)
    return o, float(m[0]), float(l[0])


def partials(q, k_cache, v_cache, block_tables, seq_lens, scale, dtype, partition_size,
             max_partitions=None, threads=None):
    """Split-K partials (m, l, o) with layouts [S,Hq,P], [S,Hq,P], [S,Hq,P,D]."""
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    block_tables = _c(block_tables, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    S, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    if max_partitions is None:
        max_partitions = max(1, -(-int(seq_lens.max(initial=0)) // partition_size))
    m = np.full((S, Hq, max_partitions), -np.inf)
    l = np.zeros((S, Hq, max_partitions))
    o = np.zeros((S, Hq, max_partitions, D))
    L = lib()
    dt = DTYPES[dtype]

    def run(r):
        L.oracle_partials(m, l, o, q, k_cache, v_cache, block_tables, seq_lens, Hq, Hkv, D,
                          BLOCK_SIZE, block_tables.shape[1], float(scale), dt,
                          partition_size, max_partitions, r[0], r[1])

    nt = threads or num_threads()
    rngs = _ranges(S, nt)
    with _cf.ThreadPoolExecutor(max(1, len(rngs))) as ex:
        list(ex.map(run, rngs))
    return m, l, o


def lse_merge(m, l, o) -> np.ndarray:
    """Merge partials of one head: m [P], l [P], o [P, D] -> [D]."""
    m = _c(m, np.float64)
    l = _c(l, np.float64)
    o = _c(o, np.float64)
    P, D = o.shape
    out = np.zeros(D, dtype=np.float64)
    lib().oracle_lse_merge(out, m, l, o, P, D)
    return out


def gather_kv(k_cache, v_cache, block_tables, s, seq_len):
    """Contiguous (K, V) of one sequence: [Hkv, seq_len, D] uint16 each."""
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    block_tables = _c(block_tables, np.int32)
    _, Hkv, _, D = k_cache.shape
    ko = np.zeros((Hkv, seq_len, D), dtype=np.uint16)
    vo = np.zeros((Hkv, seq_len, D), dtype=np.uint16)
    lib().oracle_gather_kv(ko, vo, k_cache, v_cache, block_tables, block_tables.shape[1],
                           Hkv, D, BLOCK_SIZE, s, seq_len)
    return ko, vo


def reshape_and_cache(k_cache, v_cache, k_new, v_new, slot_mapping) -> int:
    """In place on the (contiguous uint16) host pools; returns the out-of-pool count."""
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    k_new = _c(k_new, np.uint16)
    v_new = _c(v_new, np.uint16)
    slot_mapping = _c(slot_mapping, np.int64)
    nb, Hkv, _, D = k_cache.shape
    return int(lib().oracle_reshape_and_cache(k_cache, v_cache, k_new, v_new, slot_mapping,
                                              slot_mapping.shape[0], Hkv, D, BLOCK_SIZE, nb))


def copy_blocks(k_cache, v_cache, block_mapping) -> int:
    """In place on the host pools; returns the count of skipped (out-of-pool) pairs."""
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    bm = _c(block_mapping, np.int64).reshape(-1, 2)
    nb, Hkv, _, D = k_cache.shape
    return int(lib().oracle_copy_blocks(k_cache, v_cache, bm, bm.shape[0], Hkv, D,
                                        BLOCK_SIZE, nb))


def prefill(q, k_cache, v_cache, block_tables, seq_lens, query_start, scale, dtype: str,
            threads=None) -> np.ndarray:
    """Chunked-prefill output [total_rows, Hq, D] in fp64 (causal over the pool)."""
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    block_tables = _c(block_tables, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    query_start = _c(query_start, np.int32)
    T, Hq, D = q.shape
    S = seq_lens.shape[0]
    out = np.zeros((T, Hq, D), dtype=np.float64)
    L = lib()
    dt = DTYPES[dtype]

    def run(s):
        L.oracle_prefill(out, q, k_cache, v_cache, block_tables, seq_lens, query_start, Hq,
                         k_cache.shape[1], D, BLOCK_SIZE, block_tables.shape[1], float(scale), dt,
                         s, s + 1)

    nt = threads or num_threads()
    with _cf.ThreadPoolExecutor(nt) as ex:
        list(ex.map(run, range(S)))
    return out


def swap_blocks(dst_k, dst_v, src_k, src_v, block_mapping) -> int:
    """Copy blocks src (of the source pools) -> dst (of the destination pools) in place."""
    assert dst_k.flags.c_contiguous and dst_v.flags.c_contiguous
    bm = _c(block_mapping, np.int64).reshape(-1, 2)
    snb, Hkv, _, D = src_k.shape
    dnb = dst_k.shape[0]
    return int(lib().oracle_swap_blocks(dst_k, dst_v, _c(src_k, np.uint16), _c(src_v, np.uint16),
                                        bm, bm.shape[0], Hkv, D, BLOCK_SIZE, snb, dnb))


def step(w, threads=None):
    """A whole decode step of a synthetic workload on host copies of the pool.

    copy_blocks (if the workload has CoW pairs), then reshape_and_cache (if it
    appends), then decode.  Returns (out fp64, k_pool, v_pool) after the step.
    """
    k = w.k_cache.copy()
    v = w.v_cache.copy()
    if w.block_mapping is not None and len(w.block_mapping):
        copy_blocks(k, v, w.block_mapping)
    if w.slot_mapping is not None:
        reshape_and_cache(k, v, w.k_new, w.v_new, w.slot_mapping)
    out = decode(w.q, k, v, w.block_tables, w.seq_lens, w.scale, w.dtype, threads=threads)
    return out, k, v
