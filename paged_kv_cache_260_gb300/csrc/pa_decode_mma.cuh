// pa_decode_mma.cuh -- paged decode attention on the tensor cores (sm_103a).
//
// What it computes: for each sequence s and query head h,
//     out[s][h] = sum_t softmax_t(scale * q[s][h] . k_t) v_t ,  t < seq_len(s)
// with k_t, v_t read through the sequence's block table (attention over a
// KV cache kept in 16-token blocks that are not contiguous in memory; block-
// table figure of "PagedAttention：vLLM 系统论文", section 核心思想).  The score
// row is never stored: a running max and running sum rescale the partial
// result as tiles arrive (online softmax, vLLM deep notes, section
// "核心思想：Tiling + Online Softmax").  Runs cut by the work split are merged
// with the log-sum-exp rule (FlashDecoding split-K, ICML tutorial notes,
// section "内核优化").  Query heads share kv heads in groups of G
// (grouped-query attention, same notes, section "Attention 简化与 KV Cache 优化").
//
// How it maps onto GB300:
//  * Unit of data: one (physical block, kv head) tile = 16 tokens x head_dim,
//    contiguous in the pool.  K and V tiles are fetched by 2-D tensor-map TMA
//    in 64-column boxes with the 128-byte swizzle, so the fragment loads
//    below hit 8 distinct bank groups; they complete on an mbarrier.
//  * A persistent grid walks the flat (sequence, kv head, tile) list
//    (pa_schedule.cuh).  Every warp is an independent worker with its own
//    contiguous, equal share of tiles and its own ring of copy stages; warps
//    never synchronise with each other.  A run that lies in one worker's share
//    is written straight from registers; the pieces of a cut run go to
//    per-worker slots and a separate merge kernel combines them.
//  * One warp serves the whole query group of a kv head (G <= 16), so each
//    K/V byte leaves HBM once per decode.  Per tile, on the tensor cores:
//        S[16 tokens x 8 heads] = K[16 x D] . Q^T[D x 8]       (K = A operand)
//        O^T[D x 8 heads]      += V^T[D x 16] . P^T[16 x 8]    (V = A operand)
//    with mma.sync m16n8k16 and fp32 accumulation, once per 8-column tile of
//    query heads (one tile for G <= 8, two for G <= 16; each K or V fragment
//    loaded from shared memory serves both).  The group is padded to a
//    multiple of 8 columns.  P (the softmax weights, in [0, 1]) is rounded to
//    the input type for the second product and transposed in registers
//    (movmatrix), so every lane owns the same heads in S and in O: the
//    online-softmax rescale needs no data exchange between lanes.
//  * Large batches (more than kSeqsInSmem sequences) keep the per-sequence
//    lengths and unit prefix in the workspace, built once by two small
//    kernels, instead of in every block's shared memory.
#pragma once

#include <cuda.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_schedule.cuh"

namespace pa {

template <int D, int NT>
struct MmaShape {
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(NT == 1 || NT == 2, "query columns: 8 or 16");
    static constexpr int NB = D / 64;                         // 64-column boxes per tile
    static constexpr int BOX = kBlockSize * 128;              // bytes of one box (16 rows x 128 B)
    static constexpr int TILE = NB * BOX;                     // bytes of K (or V) per tile
    static constexpr int KSTEPS = D / 16;                     // QK: k-steps; PV: m-tiles
    static constexpr int QB_MAX = 8 * NT * D * 2;             // q group, up to 8 * NT heads
    static constexpr int QSLOT = (QB_MAX + 1023) / 1024 * 1024;
    static constexpr int STAGE = 2 * TILE + QSLOT;            // multiple of 1024 (swizzle atom)
};

template <int D, int NT, int W, int S>
struct MmaLayout {
    using Sh = MmaShape<D, NT>;
    static constexpr size_t stages = (size_t)W * S * Sh::STAGE;
    static constexpr size_t bars = (size_t)W * S * 8;
    // +1024: the dynamic shared memory base is aligned up to the swizzle atom
    static constexpr size_t fixed = 1024 + stages + bars;
};

// Byte offset of the 16-byte chunk `chunk` (0..7) of row `row` inside a
// 128-byte-swizzled box: chunks are permuted by the row index modulo 8.
__device__ __forceinline__ uint32_t swz(int row, int chunk)
{
    return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Row of the partial-result arrays (m, l, o) for fixed-mode partition `part`
// of run (s, h), head g: the documented [num_seqs][num_heads][P_max] layout.
__device__ __forceinline__ size_t part_row(const DecodeParams &p, int G, int s, int h, int part,
                                           int g)
{
    return ((size_t)s * p.num_heads + h * G + g) * p.p_max + part;
}

// Row of the slot arrays for worker slot `slot` (2 * worker, +1 for the
// worker's last piece), head g.
__device__ __forceinline__ size_t slot_row(int G, int slot, int g)
{
    return (size_t)slot * G + g;
}

// Large batches: the per-sequence arrays (clamped lengths, unit prefix,
// first-block-shared flags) are built once into the workspace by two kernels
// of kPrepSeqs-sequence blocks, instead of by every decode block into its
// shared memory.  decode_prep_kernel builds its block's sequences with the
// prefix counted from the block's first, and leaves the block's unit count
// and any-flag in ws_blk; decode_prep_fix_kernel adds the counts of the
// blocks before it, and its last block writes the batch's total
// (pre[num_seqs]) and whether any flag is set (share[num_seqs]).  Neither
// waits for another block of its own grid.
template <int NTH>
__global__ void __launch_bounds__(NTH) decode_prep_kernel(const DecodeParams p)
{
    static_assert(4 * NTH == kPrepSeqs, "one row of four sequences a thread per block");
    // the kernel that follows may be scheduled now; it waits for this grid
    grid_dependents_launch();
    grid_dependency_wait();
    const int begin = blockIdx.x * kPrepSeqs, end = min(p.num_seqs, begin + kPrepSeqs);
    int total;
    const bool any = __syncthreads_or(
        build_prefix<NTH, 4, 1>(p, begin, end, p.ws_pre, p.ws_lens, p.ws_share, &total));
    if (threadIdx.x == 0) {
        p.ws_blk[2 * blockIdx.x] = total;
        p.ws_blk[2 * blockIdx.x + 1] = any ? 1 : 0;
    }
}

template <int NTH>
__global__ void __launch_bounds__(NTH) decode_prep_fix_kernel(const DecodeParams p)
{
    grid_dependents_launch();
    grid_dependency_wait();
    __shared__ int red[NTH / 32][2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x, last = gridDim.x - 1;
    // the unit count of the blocks before this one (and, in the last block,
    // whether any block flagged a sequence)
    int off = 0, any = 0;
    // (written by the grid before: read through L2)
    for (int i = tid; i < b; i += NTH)
        off += __ldcg(p.ws_blk + 2 * i);
    if (b == last)
        for (int i = tid; i <= last; i += NTH)
            any |= __ldcg(p.ws_blk + 2 * i + 1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        off += __shfl_xor_sync(0xffffffffu, off, o);
        any |= __shfl_xor_sync(0xffffffffu, any, o);
    }
    if (lane == 0) {
        red[warp][0] = off;
        red[warp][1] = any;
    }
    __syncthreads();
    off = 0;
    any = 0;
#pragma unroll
    for (int w = 0; w < NTH / 32; ++w) {
        off += red[w][0];
        any |= red[w][1];
    }
    const int begin = b * kPrepSeqs, end = min(p.num_seqs, begin + kPrepSeqs);
    if (off != 0)
        for (int s = begin + tid; s < end; s += NTH)
            p.ws_pre[s] = __ldcg(p.ws_pre + s) + off;
    if (b == last && tid == 0) {
        p.ws_pre[p.num_seqs] = off + __ldcg(p.ws_blk + 2 * b);
        p.ws_share[p.num_seqs] = any ? 1 : 0;
    }
}

// L2 policy for a tile that another sequence's table also names (a block
// shared by parallel samples): normal priority, so that tiles read once
// (evict-first) leave L2 before it and the siblings' reads find it there.
__device__ __forceinline__ uint64_t l2_evict_normal_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// One warp's whole walk: its pieces, tile by tile, and their results.
// SHARE: some sequence of the batch shares its first block with a
// neighbour; only then are the neighbours' table entries looked up per tile
// (the check costs the unshared loop a few per cent even when it never
// fires, so the kernel holds two copies of the loop and picks one per block).
template <typename T, int D, int NT, int W, int S, bool SHARE, bool PARTIAL>
__device__ __forceinline__ void decode_worker(const DecodeParams &p, const CUtensorMap &tmk,
                                              const CUtensorMap &tmv, unsigned char *smem,
                                              uint64_t *bars, const int32_t *pre,
                                              const int32_t *lens, const uint8_t *share)
{
    using Sh = MmaShape<D, NT>;
    using E = Elem<T>;
    using M = Mma<T>;
    constexpr int KS = Sh::KSTEPS;
    constexpr uint32_t FULL = 0xffffffffu;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = p.num_seqs, Hkv = p.num_kv_heads, Hq = p.num_heads;
    const int G = Hq / Hkv;
    const int worker = blockIdx.x * W + warp;

    const uint64_t pol_once = l2_evict_first_policy();
    const uint64_t pol_shared = SHARE ? l2_evict_normal_policy() : pol_once;
    const uint32_t bar0 = smem_addr(&bars[warp * S]);
    unsigned char *wst = smem + (size_t)warp * S * Sh::STAGE;
    const uint32_t wst_addr = smem_addr(wst);
    const int qb_bytes = G * D * 2;

    // ---- producer: this warp's tiles, S ahead of the consumer (lane 0 issues) ----
    Walker prod;
    prod.init(pre, lens, n, Hkv, p.mode, p.part_tiles, p.min_tiles, p.workers, worker);
    Walker cons = prod;
    int ptile = prod.valid ? prod.tb : 0;
    bool pfirst = true, pdone = !prod.valid;
    // the producer's sequence shares its first block with a neighbour (read
    // once per piece, not per tile)
    bool pseq_share = SHARE && prod.valid && share[prod.s];
    auto advance = [&]() {
        while (!pdone && ptile >= prod.te) {
            prod.next();
            if (!prod.valid)
                pdone = true;
            else {
                ptile = prod.tb;
                pfirst = true;
                if constexpr (SHARE)
                    pseq_share = share[prod.s];
            }
        }
    };
    advance();
    // Physical block of the next tile and, for a sequence whose first block
    // a neighbour shares, the blocks the neighbours' tables name at the same
    // position (-1: none).  A block that a neighbour also names is shared
    // (parallel samples) and read again soon.  The loads are issued a tile
    // ahead and compared only when the tile is issued, so their latency hides
    // behind the current tile's math.
    int pphys = 0, pnb0 = -1, pnb1 = -1;
    auto lookup = [&]() {
        if (pdone || lane != 0)
            return;
        const int32_t *row = p.block_tables + (size_t)prod.s * p.max_blocks;
        pphys = __ldg(row + ptile);
        if constexpr (SHARE) {
            pnb0 = pnb1 = -1;
            if (!pseq_share)
                return;
            const int lo_tok = ptile * kBlockSize;
            if (prod.s > 0 && lens[prod.s - 1] > lo_tok)
                pnb0 = __ldg(row - p.max_blocks + ptile);
            if (prod.s + 1 < n && lens[prod.s + 1] > lo_tok)
                pnb1 = __ldg(row + p.max_blocks + ptile);
        }
    };
    lookup();
    int issued = 0;
    auto produce = [&](int st) {
        if (pdone)
            return;
        if (lane == 0) {
            int phys = pphys;
            if ((unsigned)phys >= (unsigned)p.num_blocks) {
                record_error(p.err, PA_DEVERR_TABLE_RANGE);
                phys = 0;
            }
            const int row = (phys * Hkv + prod.h) * kBlockSize;
            const uint32_t bar = bar0 + st * 8;
            const uint32_t dst = wst_addr + st * Sh::STAGE;
            uint64_t pol = pol_once;
            if constexpr (SHARE)
                pol = (pnb0 == pphys) | (pnb1 == pphys) ? pol_shared : pol_once;
            mbar_arrive_expect_tx(bar, 2 * Sh::TILE + (pfirst ? qb_bytes : 0));
#pragma unroll
            for (int b = 0; b < Sh::NB; ++b) {
                tma_load_2d(dst + b * Sh::BOX, &tmk, 64 * b, row, bar, pol);
                tma_load_2d(dst + Sh::TILE + b * Sh::BOX, &tmv, 64 * b, row, bar, pol);
            }
            if (pfirst)
                bulk_load(dst + 2 * Sh::TILE,
                          reinterpret_cast<const T *>(p.q) + ((size_t)prod.s * Hq + prod.h * G) * D,
                          qb_bytes, bar);
        }
        pfirst = false;
        ++ptile;
        advance();
        lookup();
        ++issued;
    };
#pragma unroll 1
    for (int st = 0; st < S; ++st)
        produce(st);

    // ---- per-lane fragment geometry ----
    // Query columns come in NT tiles of 8 heads; in each, lane owns heads
    // 8j + 2qd and 8j + 2qd + 1 in S and in O.
    const int r = lane >> 2;          // S: token row (and +8); O: head_dim row (and +8)
    const int qd = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;   // ldmatrix: matrix index, row within it
    const int krow = ((mi & 1) << 3) + rr, kcs = mi >> 1;   // K (A operand, row-major)
    const int vrow = ((mi >> 1) << 3) + rr, vcs = mi & 1;   // V (A operand via .trans)

    uint32_t qf[NT][KS][2];           // B fragments of Q^T for the current piece
    float o[NT][KS][4];               // O^T accumulators: (row, h0) (row, h1) (row+8, h0) (row+8, h1)
    float m[NT][2], l[NT][2];         // running max (base 2) and partial sums, heads h0, h1
    int it = 0;
    bool aborted = false;
    int abort_it = 0;
    CutDesc desc{0, 0, 0, 0, 0, 0, 0, 0};

    while (cons.valid) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            m[j][0] = m[j][1] = -INFINITY;
            l[j][0] = l[j][1] = 0.f;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    o[j][mt][c] = 0.f;
        }
        const int L = lens[cons.s];
        bool need_q = true;

        // Fused append: the new token sits at position L-1, in the run's last
        // tile, which only this warp reads.  Its K/V row is taken from
        // k_new / v_new into the stage after the tile lands (the pool slot
        // still holds a stale row) and written to the pool for later steps.
        constexpr int NCH = D / 8;                // 16-byte chunks per row
        const int last_tile = (L - 1) / kBlockSize;
        bool app = false;
        int app_phys = 0;
        uint4 app_row = make_uint4(0u, 0u, 0u, 0u);
        if (p.k_new != nullptr && L > 0 && cons.te == cons.nt) {
            const int64_t slot = __ldg(p.slot_mapping + cons.s);
            if (slot >= 0) {
                app_phys = __ldg(p.block_tables + (size_t)cons.s * p.max_blocks + last_tile);
                if ((unsigned)app_phys < (unsigned)p.num_blocks &&
                    slot == (int64_t)app_phys * kBlockSize + (L - 1) % kBlockSize) {
                    app = true;
                    if (lane < 2 * NCH) {
                        const T *src = reinterpret_cast<const T *>(lane < NCH ? p.k_new : p.v_new) +
                                       ((size_t)cons.s * Hkv + cons.h) * D + (lane % NCH) * 8;
                        app_row = __ldg(reinterpret_cast<const uint4 *>(src));
                    }
                } else if (lane == 0) {
                    record_error(p.err, PA_DEVERR_APPEND_SLOT);
                }
            }
        }

        for (int tile = cons.tb; tile < cons.te; ++tile) {
            const int st = it % S;
            if (!aborted && !mbar_wait_bounded(bar0 + st * 8, (uint32_t)((it / S) & 1))) {
                aborted = true;
                abort_it = it;
                if (lane == 0)
                    record_error(p.err, PA_DEVERR_TIMEOUT);
            }
            const uint32_t kst = wst_addr + st * Sh::STAGE;
            const uint32_t vst = kst + Sh::TILE;
            if (need_q) {
                const unsigned char *qs = wst + (size_t)st * Sh::STAGE + 2 * Sh::TILE;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int hq = 8 * j + r;     // B column: query head of the group
                    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(qs + (size_t)hq * D * 2);
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        qf[j][ks][0] = hq < G ? qrow[(16 * ks + 2 * qd) / 2] : 0u;
                        qf[j][ks][1] = hq < G ? qrow[(16 * ks + 8 + 2 * qd) / 2] : 0u;
                    }
                }
                need_q = false;
            }
            const int nvalid = min(kBlockSize, L - tile * kBlockSize);
            if (app && tile == last_tile) {
                const int row = (L - 1) % kBlockSize;
                if (lane < 2 * NCH) {
                    const int c = lane % NCH;   // chunk of 8 channels
                    unsigned char *dst = wst + (size_t)st * Sh::STAGE + (lane < NCH ? 0 : Sh::TILE) +
                                         (c >> 3) * Sh::BOX + swz(row, c & 7);
                    *reinterpret_cast<uint4 *>(dst) = app_row;
                    T *pool = reinterpret_cast<T *>(const_cast<void *>(lane < NCH ? p.k_cache : p.v_cache));
                    const size_t prow = ((size_t)app_phys * Hkv + cons.h) * kBlockSize + row;
                    *reinterpret_cast<uint4 *>(pool + prow * D + c * 8) = app_row;
                    // the next copy into this stage must not overtake these writes
                    fence_proxy_async_shared();
                }
                __syncwarp();
            }

            // S = K . Q^T  (two accumulators per column tile to shorten the
            // dependency chain; each K fragment serves every column tile)
            float sa[NT][4], sb[NT][4];
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    sa[j][c] = sb[j][c] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t a[4];
                ldsm_x4(kst + (ks >> 2) * Sh::BOX + swz(krow, 2 * (ks & 3) + kcs), a[0], a[1], a[2], a[3]);
#pragma unroll
                for (int j = 0; j < NT; ++j)
                    M::run((ks & 1) ? sb[j] : sa[j], a, qf[j][ks][0], qf[j][ks][1]);
            }
            const bool masked = nvalid < kBlockSize;
            uint32_t pb[NT][2];
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                float x0 = (sa[j][0] + sb[j][0]) * p.scale_log2;   // token r,   head h0
                float x1 = (sa[j][1] + sb[j][1]) * p.scale_log2;   // token r,   head h1
                float x2 = (sa[j][2] + sb[j][2]) * p.scale_log2;   // token r+8, head h0
                float x3 = (sa[j][3] + sb[j][3]) * p.scale_log2;   // token r+8, head h1
                if (masked) {
                    // slots past the end may hold anything, NaN included
                    if (r >= nvalid)
                        x0 = x1 = -INFINITY;
                    if (r + 8 >= nvalid)
                        x2 = x3 = -INFINITY;
                }
                float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(FULL, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(FULL, mx1, off));
                }
                if (__any_sync(FULL, (mx0 > m[j][0]) | (mx1 > m[j][1]))) {
                    const float n0 = fmaxf(m[j][0], mx0), n1 = fmaxf(m[j][1], mx1);
                    const float a0 = exp2f(m[j][0] - n0), a1 = exp2f(m[j][1] - n1);
                    m[j][0] = n0;
                    m[j][1] = n1;
                    l[j][0] *= a0;
                    l[j][1] *= a1;
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        o[j][mt][0] *= a0;
                        o[j][mt][1] *= a1;
                        o[j][mt][2] *= a0;
                        o[j][mt][3] *= a1;
                    }
                }
                const float p0 = exp2f(x0 - m[j][0]), p1 = exp2f(x1 - m[j][1]);
                const float p2 = exp2f(x2 - m[j][0]), p3 = exp2f(x3 - m[j][1]);
                l[j][0] += p0 + p2;
                l[j][1] += p1 + p3;
                // P^T as the B operand: rows of P (tokens) become columns
                pb[j][0] = movmatrix_trans(M::pack(p0, p1));
                pb[j][1] = movmatrix_trans(M::pack(p2, p3));
            }

            // O^T += V^T . P^T ; value rows past the end are zeroed (0 * NaN is NaN)
            uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
            if (masked) {
                mlo = (2 * qd < nvalid ? 0x0000ffffu : 0u) | (2 * qd + 1 < nvalid ? 0xffff0000u : 0u);
                mhi = (8 + 2 * qd < nvalid ? 0x0000ffffu : 0u) |
                      (9 + 2 * qd < nvalid ? 0xffff0000u : 0u);
            }
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                uint32_t a[4];
                ldsm_x4_trans(vst + (mt >> 2) * Sh::BOX + swz(vrow, 2 * (mt & 3) + vcs), a[0], a[1],
                              a[2], a[3]);
                a[0] &= mlo;
                a[1] &= mlo;
                a[2] &= mhi;
                a[3] &= mhi;
#pragma unroll
                for (int j = 0; j < NT; ++j)
                    M::run(o[j][mt], a, pb[j][0], pb[j][1]);
            }
            __syncwarp();
            if (!aborted)
                produce(st);
            ++it;
        }

        // ---- end of piece: write this warp's result ----
        const int s = cons.s, h = cons.h;
        const bool whole = cons.whole_run();
        const bool wp = !whole && cons.whole_part();
        const int slot = 2 * worker + (cons.first ? 0 : 1);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l[j][0] += __shfl_xor_sync(FULL, l[j][0], off);
                l[j][1] += __shfl_xor_sync(FULL, l[j][1], off);
            }
            const float inv0 = 1.f / l[j][0], inv1 = 1.f / l[j][1];
            const int h0 = 8 * j + 2 * qd, h1 = h0 + 1;
            if (PARTIAL && whole) {
                // partial-output mode: m, l and the normalised result, fp32
                const size_t row0 = (size_t)s * Hq + h * G + h0, row1 = row0 + 1;
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    const int d0 = 16 * mt + r;
                    if (h0 < G) {
                        p.out_o[row0 * D + d0] = o[j][mt][0] * inv0;
                        p.out_o[row0 * D + d0 + 8] = o[j][mt][2] * inv0;
                    }
                    if (h1 < G) {
                        p.out_o[row1 * D + d0] = o[j][mt][1] * inv1;
                        p.out_o[row1 * D + d0 + 8] = o[j][mt][3] * inv1;
                    }
                }
                if (r == 0) {
                    if (h0 < G) {
                        p.out_m[row0] = m[j][0] * kLn2;
                        p.out_l[row0] = l[j][0];
                    }
                    if (h1 < G) {
                        p.out_m[row1] = m[j][1] * kLn2;
                        p.out_l[row1] = l[j][1];
                    }
                }
            } else if (whole) {
                T *out = reinterpret_cast<T *>(p.out) + ((size_t)s * Hq + h * G) * D;
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    const int d0 = 16 * mt + r;
                    if (h0 < G) {
                        out[h0 * D + d0] = E::from_f(o[j][mt][0] * inv0);
                        out[h0 * D + d0 + 8] = E::from_f(o[j][mt][2] * inv0);
                    }
                    if (h1 < G) {
                        out[h1 * D + d0] = E::from_f(o[j][mt][1] * inv1);
                        out[h1 * D + d0 + 8] = E::from_f(o[j][mt][3] * inv1);
                    }
                }
            } else {
                // a partition (fixed mode) goes to its documented row; a cut
                // piece to this worker's first or last slot
                float *pm = wp ? p.ws_m : p.ws_sm;
                float *pl = wp ? p.ws_l : p.ws_sl;
                float *po = wp ? p.ws_o : p.ws_so;
                const size_t row0 = wp ? part_row(p, G, s, h, cons.part, h0) : slot_row(G, slot, h0);
                const size_t row1 = wp ? part_row(p, G, s, h, cons.part, h1) : slot_row(G, slot, h1);
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    const int d0 = 16 * mt + r;
                    if (h0 < G) {
                        po[row0 * D + d0] = o[j][mt][0] * inv0;
                        po[row0 * D + d0 + 8] = o[j][mt][2] * inv0;
                    }
                    if (h1 < G) {
                        po[row1 * D + d0] = o[j][mt][1] * inv1;
                        po[row1 * D + d0 + 8] = o[j][mt][3] * inv1;
                    }
                }
                if (r == 0) {
                    if (h0 < G) {
                        pm[row0] = m[j][0] * kLn2;
                        pl[row0] = l[j][0];
                    }
                    if (h1 < G) {
                        pm[row1] = m[j][1] * kLn2;
                        pl[row1] = l[j][1];
                    }
                }
            }
        }
        if (PARTIAL && whole && p.cut_of_run && lane == 0)
            reinterpret_cast<int2 *>(p.cut_of_run)[(size_t)s * p.num_kv_heads + h] =
                make_int2(-1, 0);
        if (!whole) {
            // the unit (run, or partition in fixed mode) this piece belongs to
            const int u0 = cons.F + (p.mode == kModeFixed ? cons.part * cons.pt : 0);
            const int nu = p.mode == kModeFixed ? min(cons.pt, cons.nt - cons.part * cons.pt) : cons.nt;
            if (!wp && u0 >= cons.A && u0 + nu > cons.B) {
                if (PARTIAL && p.cut_of_run && lane == 0)
                    reinterpret_cast<int2 *>(p.cut_of_run)[(size_t)s * p.num_kv_heads + h] =
                        make_int2(worker, 2 * cut_last_worker(u0, nu, cons.R) +
                                              (u0 != worker * cons.R ? 1 : 0));
                desc.s = s;
                desc.h = h;
                desc.part = cons.part;
                desc.u0 = u0;
                desc.nu = nu;
                desc.R = cons.R;
                desc.np = p.mode == kModeFixed ? (cons.nt + cons.pt - 1) / cons.pt : 1;
                desc.valid = 1;
            }
        }
        cons.next();
    }
    // every worker leaves a descriptor, valid or not, so none is stale
    if (p.ws_desc && lane == 0)
        p.ws_desc[worker] = desc;

    // a wait that gave up leaves copies in flight: let them land (bounded)
    if (aborted) {
        for (int x = abort_it; x < issued; ++x)
            mbar_wait_bounded(bar0 + (x % S) * 8, (uint32_t)((x / S) & 1));
    }
}

template <typename T, int D, int NT, int W, int S, bool PARTIAL>
__global__ void __launch_bounds__(W * 32)
decode_mma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv)
{
    using Lay = MmaLayout<D, NT, W, S>;
    using E = Elem<T>;

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::stages);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = p.num_seqs, Hq = p.num_heads;
    const bool seq_global = p.ws_pre != nullptr;

    if (lane == 0) {
        for (int st = 0; st < S; ++st)
            mbar_init(smem_addr(&bars[warp * S + st]), 1);
        mbar_init_fence();
    }
    // the merge kernels that follow may be scheduled now; they wait for us
    grid_dependents_launch();
    if (!seq_global)
        for (int i = tid * 32; i < n; i += W * 32 * 32)
            prefetch_l2(p.seq_lens + i);
    // no global memory is read or written before the preceding kernel has
    // completed (the prefetch above only warms L2)
    grid_dependency_wait();
    const int32_t *pre, *lens;
    const uint8_t *share;
    bool any_share = false;
    if (seq_global) {
        // built by decode_prep_kernel, the grid this one waited for, which
        // leaves after the flags whether any is set
        pre = p.ws_pre;
        lens = p.ws_lens;
        share = p.ws_share;
        any_share = __syncthreads_or(tid == 0 && share[n] != 0);
    } else {
        int32_t *spre = reinterpret_cast<int32_t *>(bars + W * S);
        int32_t *slens = spre + n + 1;
        uint8_t *sshare = reinterpret_cast<uint8_t *>(slens + n);
        // the barrier also publishes the arrays
        int total;
        any_share = __syncthreads_or(build_prefix<W * 32, 1, 4>(p, 0, n, spre, slens, sshare,
                                                                   &total));
        if (tid == 0)
            spre[n] = total;
        __syncthreads();
        pre = spre;
        lens = slens;
        share = sshare;
    }

    // sequences without tokens get zeros (no piece ever covers them); in
    // partial-output mode an empty partial result (m = -inf, l = 0)
    for (int s = blockIdx.x; s < n; s += gridDim.x) {
        if (lens[s] == 0) {
            if (PARTIAL) {
                for (int e = tid; e < Hq * D; e += W * 32)
                    p.out_o[(size_t)s * Hq * D + e] = 0.f;
                for (int e = tid; e < Hq; e += W * 32) {
                    p.out_m[(size_t)s * Hq + e] = -INFINITY;
                    p.out_l[(size_t)s * Hq + e] = 0.f;
                }
                if (p.cut_of_run)
                    for (int e = tid; e < p.num_kv_heads; e += W * 32)
                        reinterpret_cast<int2 *>(p.cut_of_run)[(size_t)s * p.num_kv_heads + e] =
                            make_int2(-1, 0);
            } else {
                T *o = reinterpret_cast<T *>(p.out) + (size_t)s * Hq * D;
                for (int e = tid; e < Hq * D; e += W * 32)
                    o[e] = E::from_f(0.f);
            }
        }
    }

    if (any_share)
        decode_worker<T, D, NT, W, S, true, PARTIAL>(p, tmk, tmv, smem, bars, pre, lens, share);
    else
        decode_worker<T, D, NT, W, S, false, PARTIAL>(p, tmk, tmv, smem, bars, pre, lens, share);
}

// ---------------------------------------------------------------------------
// Log-sum-exp merge of partial results (m_p, l_p, o_p):
//     M = max_p m_p,  w_p = l_p exp(m_p - M),  out = sum_p w_p o_p / sum_p w_p
// (split-K along the sequence, FlashDecoding, ICML tutorial notes, section
// "内核优化").  merge_cut_kernel combines the pieces of each cut unit: one
// thread block per worker, whose descriptor names the unit starting in its
// range; warp g takes query head g of the group, each lane D/32 channels,
// folding the pieces in one pass with a running maximum.  The result is the
// output (a run) or, in fixed mode, the partition's documented row.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(512) merge_cut_kernel(const DecodeParams p)
{
    constexpr int V = D / 32;
    constexpr int CH = 8;
    grid_dependents_launch();
    grid_dependency_wait();
    const CutDesc *dp = p.ws_desc + blockIdx.x;
    const int valid = __ldcg(&dp->valid);
    const int Hkv = p.num_kv_heads, Hq = p.num_heads, G = Hq / Hkv;
    const int g = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (!valid || g >= G)
        return;
    const int s = __ldcg(&dp->s), h = __ldcg(&dp->h), part = __ldcg(&dp->part);
    const int u0 = __ldcg(&dp->u0), nu = __ldcg(&dp->nu), R = __ldcg(&dp->R), np = __ldcg(&dp->np);
    const int c0 = blockIdx.x, c1 = cut_last_worker(u0, nu, R);
    const int npieces = c1 - c0 + 1;

    float Mx = -INFINITY, Ws = 0.f, acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v)
        acc[v] = 0.f;
    for (int base = 0; base < npieces; base += CH) {
        float mv[CH], lv[CH], ov[CH][V];
#pragma unroll
        for (int i = 0; i < CH; ++i) {
            if (base + i < npieces) {
                const int c = c0 + base + i;
                const size_t row = slot_row(G, cut_piece_slot(c, c0, u0 != c0 * R), g);
                mv[i] = __ldcg(p.ws_sm + row);
                lv[i] = __ldcg(p.ws_sl + row);
                const float *src = p.ws_so + row * D + lane * V;
                if constexpr (V == 4) {
                    const float4 x = __ldcg(reinterpret_cast<const float4 *>(src));
                    ov[i][0] = x.x, ov[i][1] = x.y, ov[i][2] = x.z, ov[i][3] = x.w;
                } else {
                    const float2 x = __ldcg(reinterpret_cast<const float2 *>(src));
                    ov[i][0] = x.x, ov[i][1] = x.y;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < CH; ++i) {
            if (base + i < npieces) {
                const float nM = fmaxf(Mx, mv[i]);
                const float a = Mx == -INFINITY ? 0.f : exp2f((Mx - nM) * kLog2e);
                const float b = lv[i] * exp2f((mv[i] - nM) * kLog2e);
                Ws = Ws * a + b;
#pragma unroll
                for (int v = 0; v < V; ++v)
                    acc[v] = acc[v] * a + b * ov[i][v];
                Mx = nM;
            }
        }
    }
    const float inv = 1.f / Ws;
    if (p.mode == kModeFixed && np >= 2) {
        const size_t row = part_row(p, G, s, h, part, g);
        float *dst = p.ws_o + row * D + lane * V;
#pragma unroll
        for (int v = 0; v < V; ++v)
            dst[v] = acc[v] * inv;
        if (lane == 0) {
            p.ws_m[row] = Mx;
            p.ws_l[row] = Ws;
        }
    } else if (p.out_o) {
        const size_t row = (size_t)s * Hq + h * G + g;
        float *dst = p.out_o + row * D + lane * V;
#pragma unroll
        for (int v = 0; v < V; ++v)
            dst[v] = acc[v] * inv;
        if (lane == 0) {
            p.out_m[row] = Mx;
            p.out_l[row] = Ws;
        }
    } else {
        using M = Mma<T>;
        T *dst = reinterpret_cast<T *>(p.out) + ((size_t)s * Hq + h * G + g) * D + lane * V;
        uint32_t *d32 = reinterpret_cast<uint32_t *>(dst);
#pragma unroll
        for (int v = 0; v < V; v += 2)
            d32[v / 2] = M::pack(acc[v] * inv, acc[v + 1] * inv);
    }
}

// Fixed mode: merge the partitions of every run with two or more of them.
// One thread block of sixteen warps per (sequence, kv head, query head of the
// group): warp w folds partitions w, w+16, ... with each lane holding D/32
// channels and eight partition rows in flight; the partial sums are added in
// shared memory.
template <typename T, int D>
__global__ void __launch_bounds__(512) merge_part_kernel(const DecodeParams p)
{
    using E = Elem<T>;
    constexpr int V = D / 32;
    constexpr int U = 8;
    constexpr int NW = 16;
    __shared__ float red_m[NW], red_w[NW];
    __shared__ float part_acc[NW][D];
    grid_dependency_wait();
    const int Hkv = p.num_kv_heads, Hq = p.num_heads, G = Hq / Hkv;
    const int g = blockIdx.x % G, run = blockIdx.x / G;
    const int s = run / Hkv, h = run % Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int L = __ldg(p.seq_lens + s);
    L = max(0, min(L, p.max_blocks * kBlockSize));
    const int nt = (L + kBlockSize - 1) / kBlockSize;
    const int np = (nt + p.part_tiles - 1) / p.part_tiles;
    if (np <= 1)
        return;
    const size_t row0 = part_row(p, G, s, h, 0, g);   // partitions of (s, h, g) are consecutive rows

    // M = max_p m_p, W = sum_p l_p exp(m_p - M)
    float Mx = -INFINITY;
    for (int pi = tid; pi < np; pi += NW * 32)
        Mx = fmaxf(Mx, __ldcg(p.ws_m + row0 + pi));
#pragma unroll
    for (int off = 16; off; off >>= 1)
        Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, off));
    if (lane == 0)
        red_m[warp] = Mx;
    __syncthreads();
    Mx = red_m[0];
#pragma unroll
    for (int w = 1; w < NW; ++w)
        Mx = fmaxf(Mx, red_m[w]);

    float acc[V], Wt = 0.f;
#pragma unroll
    for (int v = 0; v < V; ++v)
        acc[v] = 0.f;
    for (int base = warp; base < np; base += NW * U) {
        float wv[U], ov[U][V];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int pi = base + NW * u;
            if (pi < np) {
                const size_t row = row0 + pi;
                wv[u] = __ldcg(p.ws_l + row) * exp2f((__ldcg(p.ws_m + row) - Mx) * kLog2e);
                const float *src = p.ws_o + row * D + lane * V;
                if constexpr (V == 4) {
                    const float4 x = __ldcg(reinterpret_cast<const float4 *>(src));
                    ov[u][0] = x.x, ov[u][1] = x.y, ov[u][2] = x.z, ov[u][3] = x.w;
                } else {
                    const float2 x = __ldcg(reinterpret_cast<const float2 *>(src));
                    ov[u][0] = x.x, ov[u][1] = x.y;
                }
            } else {
                wv[u] = 0.f;
#pragma unroll
                for (int v = 0; v < V; ++v)
                    ov[u][v] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            Wt += wv[u];
#pragma unroll
            for (int v = 0; v < V; ++v)
                acc[v] += wv[u] * ov[u][v];
        }
    }
#pragma unroll
    for (int v = 0; v < V; ++v)
        part_acc[warp][lane * V + v] = acc[v];
    if (lane == 0)
        red_w[warp] = Wt;
    __syncthreads();
    if (tid < D) {
        float o = 0.f, W = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            o += part_acc[w][tid];
            W += red_w[w];
        }
        T *out = reinterpret_cast<T *>(p.out);
        out[((size_t)s * Hq + h * G + g) * D + tid] = E::from_f(o / W);
    }
}

template <typename T, int D, int NT>
inline void fill_kernel_set(KernelSet *ks)
{
    // one thread block per SM of W independent warps, two copy stages each.
    // At D=128 with 8 columns, 7 warps: a sweep of 6 to 10 (and 6 warps of
    // three stages) measured 7 fastest on the batch-128 GQA, long-context
    // and MHA decodes -- fewer bytes in flight per SM leave the SMs'
    // shares of HBM more even.  Otherwise as many warps as fit in shared
    // memory with the per-sequence arrays of kSeqsInSmem sequences (a
    // 16-column query slot costs two warps at D=128).
    constexpr int S = 2;
    constexpr int W = D == 128 ? (NT == 1 ? 7 : 8) : 12;
    ks->decode = reinterpret_cast<const void *>(&decode_mma_kernel<T, D, NT, W, S, false>);
    // partial outputs (m, l, normalised o: the shared-prefix decode's suffixes)
    ks->decode_partial = reinterpret_cast<const void *>(&decode_mma_kernel<T, D, NT, W, S, true>);
    ks->warps = W;
    ks->smem_fixed = MmaLayout<D, NT, W, S>::fixed;
    ks->prep = reinterpret_cast<const void *>(&decode_prep_kernel<kPrepThreads>);
    ks->prep_fix = reinterpret_cast<const void *>(&decode_prep_fix_kernel<kPrepThreads>);
    ks->merge_cut = reinterpret_cast<const void *>(&merge_cut_kernel<T, D>);
    ks->merge_part = reinterpret_cast<const void *>(&merge_part_kernel<T, D>);
}

template <typename T, int NT>
inline bool kernels_for_nt(int head_dim, KernelSet *ks)
{
    if (head_dim == 128) {
        fill_kernel_set<T, 128, NT>(ks);
        return true;
    }
    if (head_dim == 64) {
        fill_kernel_set<T, 64, NT>(ks);
        return true;
    }
    return false;
}

}  // namespace pa
