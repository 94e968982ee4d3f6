"""Seeded synthetic workloads for paged decode attention.

This module only *draws inputs*: sequence lengths, a physical block layout
(block tables over a randomly permuted pool), q / K / V values, the slots of
the appended tokens and the copy-on-write pairs.  It holds none of the
method's arithmetic (no attention, no cache writes, no copies), so both the
fp64 oracle and the CUDA path can consume the same inputs without sharing
any code that computes results.

Values are raw 16-bit patterns (``numpy.uint16``) plus a dtype tag, because
the oracle decodes fp16 / bf16 bits itself and the GPU path reinterprets the
same bits as ``torch.float16`` / ``torch.bfloat16``.

The five workloads follow the problem statement of the vLLM paper as the
reading notes "PagedAttention：vLLM 系统论文" retell it (16-token blocks
addressed through per-sequence block tables over a pool allocated once:
block-pool figure in section 核心思想, section 系统实现要点), with grouped-query
heads as in the ICML tutorial notes (section "Attention 简化与 KV Cache 优化").
Their sizes:

==========  =====  =======  ===  =====  =======================================
name        seqs   Hq/Hkv   D    dtype  lengths (post-append)
==========  =====  =======  ===  =====  =======================================
tiny        4      8/8      64   f16    U[1,100], 64-block pool, +1 token
mha7b       64     32/32    128  f16    U[512,2048]
gqa8b       128    32/8     128  bf16   lognormal(ln 600, 1) clipped [16,4096],
                                         +1 token via slot_mapping
long        4      32/8     128  bf16   {32768, 65536, 98304, 131072},
                                         512-token split-K partitions
parsamp     16x8   40/8     128  f16    1024 shared + U[0,256] + 1,
                                         copy-on-write of the last shared block
batch20k    20000  32/2     128  bf16   U[1,256], +1 token (a large batch at
                                         group 16; not one of the five)
==========  =====  =======  ===  =====  =======================================
"""
from __future__ import annotations

import concurrent.futures as _cf
import math
import os
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

BLOCK_SIZE = 16

F16 = "f16"
BF16 = "bf16"
DTYPE_CODE = {F16: 0, BF16: 1}
# quiet-NaN bit patterns, used to poison pool slots that hold no live token
NAN_BITS = {F16: 0x7E00, BF16: 0x7FC0}


# ----------------------------------------------------------------------------
# fp32 -> 16-bit conversion of drawn values (round to nearest even)
# ----------------------------------------------------------------------------
def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp32 draws to fp16 / bf16 (RNE) and return the raw bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        import torch
        t = torch.from_numpy(x).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16)
    raise ValueError(dtype)


def _normal_bits(seed_seq: np.random.SeedSequence, n: int, dtype: str,
                 chunk: int = 1 << 23) -> np.ndarray:
    """n standard-normal draws as 16-bit patterns.

    Drawn in fixed-size chunks, each from its own child of ``seed_seq``, so the
    result does not depend on how many threads produce it.
    """
    out = np.empty(n, dtype=np.uint16)
    nchunks = max(1, (n + chunk - 1) // chunk)
    children = seed_seq.spawn(nchunks)

    def work(i):
        lo = i * chunk
        hi = min(n, lo + chunk)
        if hi <= lo:
            return
        g = np.random.Generator(np.random.PCG64(children[i]))
        out[lo:hi] = to_bits(g.standard_normal(hi - lo, dtype=np.float32), dtype)

    if nchunks == 1:
        work(0)
    else:
        nthreads = min(nchunks, max(1, len(os.sched_getaffinity(0))))
        with _cf.ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(work, range(nchunks)))
    return out


# ----------------------------------------------------------------------------
# workload description
# ----------------------------------------------------------------------------
@dataclass
class Workload:
    """One decode step's inputs, in the library's layouts.

    q              [num_seqs, Hq, D]            uint16 bits
    k_cache/v_cache[num_blocks, Hkv, 16, D]     uint16 bits (state *before* the step)
    block_tables   [num_seqs, max_blocks] int32 (tables the decode reads; -1 = unused)
    seq_lens       [num_seqs] int32              post-append lengths
    k_new/v_new    [num_tokens, Hkv, D] uint16   tokens written by reshape_and_cache
    slot_mapping   [num_tokens] int64            slot = block * 16 + offset, <0 = skip
    block_mapping  [num_pairs, 2] int64          (src, dst) pairs for copy_blocks
    tables_before_cow  tables before the copy-on-write remap (None if no CoW)
    live           [num_blocks, 16] bool         slots holding a live token after the step
    """

    name: str
    dtype: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    scale: float
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    block_tables: np.ndarray
    seq_lens: np.ndarray
    k_new: Optional[np.ndarray] = None
    v_new: Optional[np.ndarray] = None
    slot_mapping: Optional[np.ndarray] = None
    block_mapping: Optional[np.ndarray] = None
    tables_before_cow: Optional[np.ndarray] = None
    live: Optional[np.ndarray] = None
    partition_size: int = 0
    query_start: Optional[np.ndarray] = None   # prefill: rows of q per sequence [S+1]
    meta: dict = field(default_factory=dict)

    @property
    def num_blocks(self) -> int:
        return self.k_cache.shape[0]

    @property
    def max_blocks_per_seq(self) -> int:
        return self.block_tables.shape[1]

    @property
    def dtype_code(self) -> int:
        return DTYPE_CODE[self.dtype]

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads

    def kv_read_bytes(self) -> int:
        """Bytes of K and V one decode step must read (every live token, every kv head)."""
        return kv_bytes(int(self.seq_lens.astype(np.int64).sum()), 1,
                        self.num_kv_heads * self.head_dim, 2)

    def unique_kv_read_bytes(self) -> int:
        """Like kv_read_bytes but counting each physical block once (shared prefixes)."""
        seen = {}
        for s in range(self.num_seqs):
            L = int(self.seq_lens[s])
            for b in range((L + BLOCK_SIZE - 1) // BLOCK_SIZE):
                phys = int(self.block_tables[s, b])
                n = min(BLOCK_SIZE, L - b * BLOCK_SIZE)
                seen[phys] = max(seen.get(phys, 0), n)
        toks = sum(seen.values())
        return kv_bytes(toks, 1, self.num_kv_heads * self.head_dim, 2)


def kv_bytes(num_tokens: int, num_layers: int, kv_width: int, dtype_bytes: int) -> int:
    """KV-cache bytes: K and V, per layer, per token, ``kv_width`` = heads x head_dim.

    Same accounting as the worked example of the mlsys-02 course page
    (section 6 练习与要点, 例 1): 2 x layers x hidden x tokens x bytes.
    """
    return 2 * num_layers * kv_width * num_tokens * dtype_bytes


def cdiv(a: int, b: int) -> int:
    return (a + b - 1) // b


# ----------------------------------------------------------------------------
# generic builder
# ----------------------------------------------------------------------------
def _layout(rng, seq_lens, num_blocks_needed, pool_blocks, max_blocks):
    """Place each sequence's logical blocks on a random permutation of the pool."""
    perm = rng.permutation(pool_blocks).astype(np.int32)
    tables = np.full((len(seq_lens), max_blocks), -1, dtype=np.int32)
    i = 0
    for s, L in enumerate(seq_lens):
        nb = cdiv(int(L), BLOCK_SIZE)
        tables[s, :nb] = perm[i:i + nb]
        i += nb
    assert i == num_blocks_needed
    return tables, perm[num_blocks_needed:]


def _live_mask(tables, seq_lens, pool_blocks):
    live = np.zeros((pool_blocks, BLOCK_SIZE), dtype=bool)
    for s, L in enumerate(seq_lens):
        L = int(L)
        for b in range(cdiv(L, BLOCK_SIZE)):
            n = min(BLOCK_SIZE, L - b * BLOCK_SIZE)
            live[tables[s, b], :n] = True
    return live


def _poison(cache, live, dtype):
    """Fill every slot that holds no live token with NaN (all kv heads)."""
    by_slot = cache.transpose(0, 2, 1, 3)          # [block, slot, kv head, d] view
    by_slot[~live] = NAN_BITS[dtype]


def build(name: str, num_seqs: int, num_heads: int, num_kv_heads: int,
          head_dim: int, dtype: str, seq_lens, seed: int, *,
          pool_blocks: Optional[int] = None, pool_factor: float = 1.25,
          append: bool = False, poison: bool = False, partition_size: int = 0,
          max_blocks: Optional[int] = None, scale: Optional[float] = None,
          table_fill: int = -1) -> Workload:
    """A decode step over ``seq_lens`` (post-append) in a randomly placed pool.

    ``append``: the last token of every sequence is the step's new token.  It is
    supplied in k_new / v_new with its slot in slot_mapping; its pool slot holds
    a stale value (NaN when ``poison``) until reshape_and_cache writes it.
    """
    ss = np.random.SeedSequence(seed)
    s_layout, s_q, s_k, s_v, s_new = ss.spawn(5)
    rng = np.random.Generator(np.random.PCG64(s_layout))
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    assert seq_lens.shape == (num_seqs,)
    needed = int(sum(cdiv(int(L), BLOCK_SIZE) for L in seq_lens))
    if pool_blocks is None:
        pool_blocks = max(1, int(math.ceil(pool_factor * needed)))
    assert pool_blocks >= needed
    if max_blocks is None:
        max_blocks = max(1, cdiv(int(seq_lens.max(initial=0)), BLOCK_SIZE))
    tables, _ = _layout(rng, seq_lens, needed, pool_blocks, max_blocks)
    if table_fill != -1:
        tables[tables < 0] = table_fill
    D, Hq, Hkv = head_dim, num_heads, num_kv_heads
    q = _normal_bits(s_q, num_seqs * Hq * D, dtype).reshape(num_seqs, Hq, D)
    k = _normal_bits(s_k, pool_blocks * Hkv * BLOCK_SIZE * D, dtype).reshape(
        pool_blocks, Hkv, BLOCK_SIZE, D)
    v = _normal_bits(s_v, pool_blocks * Hkv * BLOCK_SIZE * D, dtype).reshape(
        pool_blocks, Hkv, BLOCK_SIZE, D)
    live = _live_mask(tables, seq_lens, pool_blocks)
    w = Workload(name, dtype, num_seqs, Hq, Hkv, D,
                 1.0 / math.sqrt(D) if scale is None else scale,
                 q, k, v, tables, seq_lens, live=live,
                 partition_size=partition_size)
    if append:
        nl = _normal_bits(s_new, 2 * num_seqs * Hkv * D, dtype).reshape(2, num_seqs, Hkv, D)
        w.k_new = np.ascontiguousarray(nl[0])
        w.v_new = np.ascontiguousarray(nl[1])
        slots = np.full(num_seqs, -1, dtype=np.int64)
        for s, L in enumerate(seq_lens):
            L = int(L)
            if L > 0:
                pos = L - 1
                slots[s] = int(tables[s, pos // BLOCK_SIZE]) * BLOCK_SIZE + pos % BLOCK_SIZE
        w.slot_mapping = slots
        if poison:
            # the slot the new token goes to is stale before the write
            stale = live.copy()
            for sl in slots:
                if sl >= 0:
                    stale[sl // BLOCK_SIZE, sl % BLOCK_SIZE] = False
            _poison(k, stale, dtype)
            _poison(v, stale, dtype)
    elif poison:
        _poison(k, live, dtype)
        _poison(v, live, dtype)
    return w


# ----------------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------------
def lens_tiny(rng):
    return rng.integers(1, 100, size=4, endpoint=True)


def lens_mha7b(rng, n=64):
    return rng.integers(512, 2048, size=n, endpoint=True)


def lens_gqa8b(rng, n=128):
    x = rng.lognormal(mean=math.log(600.0), sigma=1.0, size=n)
    return np.clip(np.rint(x), 16, 4096).astype(np.int64)


LONG_LENS = (32768, 65536, 98304, 131072)


def _len_rng(seed):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7])))


def tiny(poison=False, seed=1001):
    lens = lens_tiny(_len_rng(seed))
    return build("tiny", 4, 8, 8, 64, F16, lens, seed, pool_blocks=64,
                 append=True, poison=poison)


def mha7b(poison=False, seed=1002, num_seqs=64):
    lens = lens_mha7b(_len_rng(seed), num_seqs)
    return build("mha7b", num_seqs, 32, 32, 128, F16, lens, seed, poison=poison)


def gqa8b(poison=False, seed=1003, num_seqs=128):
    lens = lens_gqa8b(_len_rng(seed), num_seqs)
    return build("gqa8b", num_seqs, 32, 8, 128, BF16, lens, seed, append=True,
                 poison=poison)


def long(poison=False, seed=1004, lens=LONG_LENS, partition_size=512):
    return build("long", len(lens), 32, 8, 128, BF16, list(lens), seed,
                 poison=poison, partition_size=partition_size)


def parsamp(poison=False, seed=1005, num_prompts=16, samples=8, prompt_len=1024,
            max_suffix=256, num_heads=40, num_kv_heads=8, head_dim=128,
            dtype=F16, suffix_lens=None):
    """Parallel sampling: each prompt's blocks are shared by its samples.

    Every step, the last shared prompt block (logical block ``(prompt_len-1)//16``)
    is copied for samples 1..S-1 of each prompt (sample 0 keeps the original, as a
    refcount dropping to one would), those samples' tables are remapped to their
    copies, the new token of every sample is written with reshape_and_cache and
    decode runs over ``prompt_len + suffix + 1`` tokens.  With a block-aligned
    prompt the new token lands in a private suffix block; with an unaligned
    prompt and a zero suffix it lands in the (copied) shared block itself.
    """
    ss = np.random.SeedSequence(seed)
    s_len, s_layout, s_q, s_k, s_v, s_new = ss.spawn(6)
    rng = np.random.Generator(np.random.PCG64(s_len))
    S, P = samples, num_prompts
    if suffix_lens is None:
        suffix = rng.integers(0, max_suffix, size=(P, S), endpoint=True)
    else:
        suffix = np.asarray(suffix_lens, dtype=np.int64).reshape(P, S)
    lens = (prompt_len + suffix + 1).reshape(-1).astype(np.int32)
    n = P * S
    pb = cdiv(prompt_len, BLOCK_SIZE)          # prompt blocks (shared)
    last_shared = pb - 1
    # unique blocks: shared prompt blocks, the S-1 copies, private blocks
    priv = [cdiv(int(L), BLOCK_SIZE) - pb for L in lens]
    needed = P * pb + P * (S - 1) + sum(priv)
    pool_blocks = int(math.ceil(1.25 * needed))
    lrng = np.random.Generator(np.random.PCG64(s_layout))
    perm = lrng.permutation(pool_blocks).astype(np.int32)
    max_blocks = cdiv(int(lens.max()), BLOCK_SIZE)
    before = np.full((n, max_blocks), -1, dtype=np.int32)
    after = np.full((n, max_blocks), -1, dtype=np.int32)
    pairs = []
    i = 0
    for p in range(P):
        shared = perm[i:i + pb]
        i += pb
        copies = perm[i:i + S - 1]
        i += S - 1
        for smp in range(S):
            s = p * S + smp
            before[s, :pb] = shared
            after[s, :pb] = shared
            if smp > 0:
                after[s, last_shared] = copies[smp - 1]
                pairs.append((int(shared[last_shared]), int(copies[smp - 1])))
            nb = priv[s]
            before[s, pb:pb + nb] = perm[i:i + nb]
            after[s, pb:pb + nb] = perm[i:i + nb]
            i += nb
    assert i == needed
    D, Hq, Hkv = head_dim, num_heads, num_kv_heads
    q = _normal_bits(s_q, n * Hq * D, dtype).reshape(n, Hq, D)
    k = _normal_bits(s_k, pool_blocks * Hkv * BLOCK_SIZE * D, dtype).reshape(
        pool_blocks, Hkv, BLOCK_SIZE, D)
    v = _normal_bits(s_v, pool_blocks * Hkv * BLOCK_SIZE * D, dtype).reshape(
        pool_blocks, Hkv, BLOCK_SIZE, D)
    nl = _normal_bits(s_new, 2 * n * Hkv * D, dtype).reshape(2, n, Hkv, D)
    slots = np.empty(n, dtype=np.int64)
    for s, L in enumerate(lens):
        pos = int(L) - 1
        slots[s] = int(after[s, pos // BLOCK_SIZE]) * BLOCK_SIZE + pos % BLOCK_SIZE
    live = _live_mask(after, lens, pool_blocks)
    # the shared block's slots are live in the copies too; poisoning must only
    # touch slots that no table (before or after the remap) can reach
    live |= _live_mask(before, np.minimum(lens, prompt_len), pool_blocks)
    if poison:
        # stale: copies (dst of the CoW, filled by copy_blocks), new-token slots
        stale = live.copy()
        for _, dst in pairs:
            stale[dst, :] = False
        for sl in slots:
            stale[sl // BLOCK_SIZE, sl % BLOCK_SIZE] = False
        _poison(k, stale, dtype)
        _poison(v, stale, dtype)
    w = Workload("parsamp", dtype, n, Hq, Hkv, D, 1.0 / math.sqrt(D), q, k, v,
                 after, lens, k_new=np.ascontiguousarray(nl[0]),
                 v_new=np.ascontiguousarray(nl[1]), slot_mapping=slots,
                 block_mapping=np.asarray(pairs, dtype=np.int64).reshape(-1, 2),
                 tables_before_cow=before, live=live)
    w.meta.update(num_prompts=P, samples=S, prompt_len=prompt_len)
    return w


def parsamp8k(poison=False, seed=1009):
    """Parallel sampling with a long prompt: as parsamp, with 8192 prompt
    tokens (8176 of them in blocks shared by the 8 samples of a prompt)."""
    w = parsamp(poison=poison, seed=seed, prompt_len=8192)
    w.name = "parsamp8k"
    return w


def batch20k(poison=False, seed=1008, num_seqs=20000):
    """A large continuous batch: 20,000 sequences, 32 query / 2 kv heads
    (group 16), head_dim 128, bf16, lengths U[1, 256], one new token each."""
    lens = _len_rng(seed).integers(1, 256, size=num_seqs, endpoint=True)
    return build("batch20k", num_seqs, 32, 2, 128, BF16, lens, seed, append=True, poison=poison)


def build_prefill(name: str, num_heads: int, num_kv_heads: int, head_dim: int, dtype: str,
                  seq_lens, chunk_lens, seed: int, *, pool_factor: float = 1.25,
                  poison: bool = False, max_blocks: Optional[int] = None) -> Workload:
    """A chunked-prefill step: sequence s holds seq_lens[s] tokens whose last
    chunk_lens[s] are the chunk being prefilled (their K/V already in the
    pool); q has one row per chunk token, rows of sequence s starting at
    query_start[s]."""
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    chunk_lens = np.asarray(chunk_lens, dtype=np.int32)
    assert np.all(chunk_lens <= seq_lens)
    w = build(name, len(seq_lens), num_heads, num_kv_heads, head_dim, dtype, seq_lens, seed,
              pool_factor=pool_factor, poison=poison, max_blocks=max_blocks)
    qs = np.zeros(len(seq_lens) + 1, dtype=np.int32)
    qs[1:] = np.cumsum(chunk_lens)
    ss = np.random.SeedSequence([seed, 11])
    w.q = _normal_bits(ss, int(qs[-1]) * num_heads * head_dim, dtype).reshape(
        int(qs[-1]), num_heads, head_dim)
    w.query_start = qs
    return w


def prefill_chunks(seed=1006):
    """Chunked prefill, GQA-8B-shaped: 8 sequences, 32/8 heads, head_dim 128,
    bf16; contexts U[512, 4096] ending in a 512-token chunk."""
    rng = _len_rng(seed)
    lens = rng.integers(512, 4096, size=8, endpoint=True)
    return build_prefill("prefill", 32, 8, 128, BF16, lens, np.full(8, 512), seed)


def prefill_long(seed=1007):
    """Chunked prefill deep into long prompts: 16 sequences, 32/8 heads,
    head_dim 128, bf16; each 16384 tokens long, ending in a 2048-token chunk."""
    return build_prefill("prefill_long", 32, 8, 128, BF16, np.full(16, 16384), np.full(16, 2048),
                         seed)


WORKLOADS = {
    "tiny": tiny,
    "mha7b": mha7b,
    "gqa8b": gqa8b,
    "long": long,
    "parsamp": parsamp,
    "batch20k": batch20k,
    "parsamp8k": parsamp8k,
    "prefill": prefill_chunks,
    "prefill_long": prefill_long,
}


def by_name(name: str, **kw) -> Workload:
    return WORKLOADS[name](**kw)


def describe(w: Workload) -> str:
    L = w.seq_lens
    return (f"{w.name}: {w.num_seqs} seqs, Hq/Hkv {w.num_heads}/{w.num_kv_heads}, "
            f"D {w.head_dim}, {w.dtype}, lens [{int(L.min())},{int(L.max())}] "
            f"mean {float(L.mean()):.1f}, pool {w.num_blocks} blocks")
