"""Pure-Python brute force for tiny inputs (test infrastructure only).

An independent restatement of paged decode attention with Python floats:
16-bit patterns decoded with ``struct`` (IEEE half via the 'e' format, bf16
as the top half of an IEEE single), K/V fetched token by token through the
block table, scores, ``math.exp`` weights and ``math.fsum`` sums.  It exists to
pin ``oracle.c``; it is far too slow for anything but a handful of tokens.
"""
from __future__ import annotations

import math
import struct


def value(bits: int, dtype: str) -> float:
    if dtype == "f16":
        return struct.unpack("<e", struct.pack("<H", int(bits)))[0]
    return struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0]


def paged_attention(q, k_cache, v_cache, block_tables, seq_lens, scale, dtype):
    """Nested lists out[s][h][d] of Python floats."""
    num_seqs, num_heads, head_dim = len(q), len(q[0]), len(q[0][0])
    num_kv_heads = len(k_cache[0])
    block_size = len(k_cache[0][0])
    group = num_heads // num_kv_heads
    out = []
    for s in range(num_seqs):
        L = int(seq_lens[s])
        rows = []
        for h in range(num_heads):
            g = h // group
            qv = [value(x, dtype) for x in q[s][h]]
            keys, vals = [], []
            for t in range(L):
                blk = int(block_tables[s][t // block_size])
                off = t % block_size
                keys.append([value(x, dtype) for x in k_cache[blk][g][off]])
                vals.append([value(x, dtype) for x in v_cache[blk][g][off]])
            if L == 0:
                rows.append([0.0] * head_dim)
                continue
            scores = [scale * math.fsum(a * b for a, b in zip(qv, kk)) for kk in keys]
            top = max(scores)
            e = [math.exp(x - top) for x in scores]
            z = math.fsum(e)
            rows.append([math.fsum(e[t] * vals[t][d] for t in range(L)) / z
                         for d in range(head_dim)])
        out.append(rows)
    return out
