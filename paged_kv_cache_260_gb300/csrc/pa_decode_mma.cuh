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
//    (pa_schedule.cuh).  Each warp owns a ring of copy stages and takes every
//    W-th tile of its block's current run; warps combine their softmax states
//    in shared memory at the end of a run.
//  * One warp serves the whole query group of a kv head (G <= 8), so each K/V
//    byte leaves HBM once per decode.  Per tile, on the tensor cores:
//        S[16 tokens x 8 heads] = K[16 x D] . Q^T[D x 8]       (K = A operand)
//        O^T[D x 8 heads]      += V^T[D x 16] . P^T[16 x 8]    (V = A operand)
//    with mma.sync m16n8k16 and fp32 accumulation.  The group is padded to 8
//    columns.  P (the softmax weights, in [0, 1]) is rounded to the input
//    type for the second product and transposed in registers (movmatrix), so
//    every lane owns the same two heads in S and in O: the online-softmax
//    rescale needs no data exchange between lanes.
#pragma once

#include <cuda.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_schedule.cuh"

namespace pa {

template <int D>
struct MmaShape {
    static_assert(D == 64 || D == 128, "head_dim");
    static constexpr int NB = D / 64;                         // 64-column boxes per tile
    static constexpr int BOX = kBlockSize * 128;              // bytes of one box (16 rows x 128 B)
    static constexpr int TILE = NB * BOX;                     // bytes of K (or V) per tile
    static constexpr int KSTEPS = D / 16;                     // QK: k-steps; PV: m-tiles
    static constexpr int QB_MAX = 8 * D * 2;                  // q group, up to 8 heads
    static constexpr int QSLOT = (QB_MAX + 1023) / 1024 * 1024;
    static constexpr int STAGE = 2 * TILE + QSLOT;            // multiple of 1024 (swizzle atom)
};

template <int D, int W, int S>
struct MmaLayout {
    using Sh = MmaShape<D>;
    static constexpr size_t stages = (size_t)W * S * Sh::STAGE;
    static constexpr size_t cm = (size_t)W * 8 * 4;
    static constexpr size_t cl = cm;
    static constexpr size_t cacc = (size_t)W * 8 * D * 4;
    static constexpr size_t bars = (size_t)W * S * 8;
    // +1024: the dynamic shared memory base is aligned up to the swizzle atom
    static constexpr size_t fixed = 1024 + stages + cm + cl + cacc + bars;
};

// Byte offset of the 16-byte chunk `chunk` (0..7) of row `row` inside a
// 128-byte-swizzled box: chunks are permuted by the row index modulo 8.
__device__ __forceinline__ uint32_t swz(int row, int chunk)
{
    return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

template <typename T, int D, int W, int S>
__global__ void __launch_bounds__(W * 32)
decode_mma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv)
{
    using Sh = MmaShape<D>;
    using Lay = MmaLayout<D, W, S>;
    using E = Elem<T>;
    using M = Mma<T>;
    constexpr int KS = Sh::KSTEPS;
    constexpr uint32_t FULL = 0xffffffffu;

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    unsigned char *stage_base = smem;
    float *cm = reinterpret_cast<float *>(smem + Lay::stages);
    float *cl = cm + W * 8;
    float *cacc = cl + W * 8;
    uint64_t *bars = reinterpret_cast<uint64_t *>(cacc + W * 8 * D);
    int32_t *pre = reinterpret_cast<int32_t *>(bars + W * S);
    int32_t *lens = pre + p.num_seqs + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = p.num_seqs, Hkv = p.num_kv_heads, Hq = p.num_heads;
    const int G = Hq / Hkv;

    if (lane == 0) {
        for (int st = 0; st < S; ++st)
            mbar_init(smem_addr(&bars[warp * S + st]), 1);
        mbar_init_fence();
    }
    build_prefix<W>(p, pre, lens);
    __syncthreads();

    if (p.mode == kModeBalanced && blockIdx.x == 0)
        for (int s = tid; s <= n; s += W * 32)
            p.ws_prefix[s] = pre[s];
    for (int s = blockIdx.x; s < n; s += gridDim.x) {
        if (lens[s] == 0) {
            T *o = reinterpret_cast<T *>(p.out) + (size_t)s * Hq * D;
            for (int e = tid; e < Hq * D; e += W * 32)
                o[e] = E::from_f(0.f);
        }
    }

    const uint64_t pol = l2_evict_first_policy();
    const uint32_t bar0 = smem_addr(&bars[warp * S]);
    unsigned char *wst = stage_base + (size_t)warp * S * Sh::STAGE;
    const uint32_t wst_addr = smem_addr(wst);
    const int qb_bytes = G * D * 2;

    // ---- producer: this warp's tiles, S ahead of the consumer (lane 0 issues) ----
    Walker prod;
    prod.init(pre, lens, n, Hkv, p.mode, p.part_tiles, p.min_tiles, gridDim.x, blockIdx.x);
    Walker cons = prod;
    int ptile = prod.valid ? prod.tb + warp : 0;
    bool pfirst = true, pdone = !prod.valid;
    auto advance = [&]() {
        while (!pdone && ptile >= prod.te) {
            prod.next();
            if (!prod.valid)
                pdone = true;
            else {
                ptile = prod.tb + warp;
                pfirst = true;
            }
        }
    };
    advance();
    int pphys = 0;
    if (!pdone && lane == 0)
        pphys = __ldg(p.block_tables + (size_t)prod.s * p.max_blocks + ptile);
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
        ptile += W;
        advance();
        if (!pdone && lane == 0)
            pphys = __ldg(p.block_tables + (size_t)prod.s * p.max_blocks + ptile);
        ++issued;
    };
#pragma unroll 1
    for (int st = 0; st < S; ++st)
        produce(st);

    // ---- per-lane fragment geometry ----
    const int r = lane >> 2;          // S: token row (and +8); O: head_dim row (and +8)
    const int qd = lane & 3;          // S and O: heads 2*qd, 2*qd + 1
    const int h0 = 2 * qd, h1 = h0 + 1;
    const int mi = lane >> 3, rr = lane & 7;   // ldmatrix: matrix index, row within it
    const int krow = ((mi & 1) << 3) + rr, kcs = mi >> 1;   // K (A operand, row-major)
    const int vrow = ((mi >> 1) << 3) + rr, vcs = mi & 1;   // V (A operand via .trans)

    uint32_t qf[KS][2];               // B fragments of Q^T for the current piece
    float o[KS][4];                   // O^T accumulators: (row, h0) (row, h1) (row+8, h0) (row+8, h1)
    float m0, m1, l0, l1;             // running max (base 2) and partial sums, heads h0, h1
    int it = 0;
    bool aborted = false;
    int abort_it = 0;

    while (cons.valid) {
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                o[mt][c] = 0.f;
        const int L = lens[cons.s];
        bool need_q = true;

        for (int tile = cons.tb + warp; tile < cons.te; tile += W) {
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
                for (int ks = 0; ks < KS; ++ks) {
                    const uint32_t *row = reinterpret_cast<const uint32_t *>(qs + (size_t)r * D * 2);
                    qf[ks][0] = r < G ? row[(16 * ks + 2 * qd) / 2] : 0u;
                    qf[ks][1] = r < G ? row[(16 * ks + 8 + 2 * qd) / 2] : 0u;
                }
                need_q = false;
            }
            const int nvalid = min(kBlockSize, L - tile * kBlockSize);

            // S = K . Q^T  (two accumulators to shorten the dependency chain)
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t a[4];
                ldsm_x4(kst + (ks >> 2) * Sh::BOX + swz(krow, 2 * (ks & 3) + kcs), a[0], a[1], a[2], a[3]);
                M::run((ks & 1) ? sb : sa, a, qf[ks][0], qf[ks][1]);
            }
            float x0 = (sa[0] + sb[0]) * p.scale_log2;   // token r,   head h0
            float x1 = (sa[1] + sb[1]) * p.scale_log2;   // token r,   head h1
            float x2 = (sa[2] + sb[2]) * p.scale_log2;   // token r+8, head h0
            float x3 = (sa[3] + sb[3]) * p.scale_log2;   // token r+8, head h1
            const bool masked = nvalid < kBlockSize;
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
            if (__any_sync(FULL, (mx0 > m0) | (mx1 > m1))) {
                const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
                const float a0 = exp2f(m0 - n0), a1 = exp2f(m1 - n1);
                m0 = n0;
                m1 = n1;
                l0 *= a0;
                l1 *= a1;
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    o[mt][0] *= a0;
                    o[mt][1] *= a1;
                    o[mt][2] *= a0;
                    o[mt][3] *= a1;
                }
            }
            const float p0 = exp2f(x0 - m0), p1 = exp2f(x1 - m1);
            const float p2 = exp2f(x2 - m0), p3 = exp2f(x3 - m1);
            l0 += p0 + p2;
            l1 += p1 + p3;
            // P^T as the B operand: rows of P (tokens) become columns
            const uint32_t pb0 = movmatrix_trans(M::pack(p0, p1));
            const uint32_t pb1 = movmatrix_trans(M::pack(p2, p3));

            // O^T += V^T . P^T
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
                M::run(o[mt], a, pb0, pb1);
            }
            __syncwarp();
            if (!aborted)
                produce(st);
            ++it;
        }

        // ---- end of piece: combine the warps' states ----
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(FULL, l0, off);
            l1 += __shfl_xor_sync(FULL, l1, off);
        }
        if (r == 0) {
            if (h0 < G) {
                cm[warp * 8 + h0] = m0;
                cl[warp * 8 + h0] = l0;
            }
            if (h1 < G) {
                cm[warp * 8 + h1] = m1;
                cl[warp * 8 + h1] = l1;
            }
        }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            const int d0 = 16 * mt + r;
            if (h0 < G) {
                cacc[(warp * 8 + h0) * D + d0] = o[mt][0];
                cacc[(warp * 8 + h0) * D + d0 + 8] = o[mt][2];
            }
            if (h1 < G) {
                cacc[(warp * 8 + h1) * D + d0] = o[mt][1];
                cacc[(warp * 8 + h1) * D + d0 + 8] = o[mt][3];
            }
        }
        __syncthreads();
        {
            const bool whole = cons.whole();
            for (int e = tid; e < G * D; e += W * 32) {
                const int g = e / D, d = e % D;
                float Mx = -INFINITY;
#pragma unroll
                for (int w = 0; w < W; ++w)
                    Mx = fmaxf(Mx, cm[w * 8 + g]);
                float Ls = 0.f, O = 0.f;
#pragma unroll
                for (int w = 0; w < W; ++w) {
                    const float mw = cm[w * 8 + g];
                    const float f = mw == -INFINITY ? 0.f : exp2f(mw - Mx);
                    Ls += f * cl[w * 8 + g];
                    O += f * cacc[(w * 8 + g) * D + d];
                }
                const float res = O / Ls;
                if (whole) {
                    T *out = reinterpret_cast<T *>(p.out);
                    out[((size_t)cons.s * Hq + cons.h * G + g) * D + d] = E::from_f(res);
                } else {
                    size_t row;
                    if (p.mode == kModeBalanced)
                        row = (size_t)(2 * blockIdx.x + (cons.first ? 0 : 1)) * G + g;
                    else
                        row = ((size_t)cons.s * Hq + cons.h * G + g) * p.p_max + cons.part;
                    p.ws_o[row * D + d] = res;
                    if (d == 0) {
                        p.ws_m[row] = Mx * kLn2;
                        p.ws_l[row] = Ls;
                    }
                }
            }
        }
        __syncthreads();
        cons.next();
    }

    // a wait that gave up leaves copies in flight: let them land (bounded)
    if (aborted) {
        for (int x = abort_it; x < issued; ++x)
            mbar_wait_bounded(bar0 + (x % S) * 8, (uint32_t)((x / S) & 1));
    }
}

// ---------------------------------------------------------------------------
// Log-sum-exp merge of split runs (the rule the split-K partials obey):
//     M = max_p m_p,  w_p = l_p exp(m_p - M),  out = sum_p w_p o_p / sum_p w_p.
// One thread block per (sequence, kv head); runs that were not cut return.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(128) merge_kernel(const DecodeParams p)
{
    using E = Elem<T>;
    constexpr int CH = 64;            // pieces whose weights are staged at a time
    __shared__ float sM[8], sW[8];
    __shared__ float wts[CH][8];
    const int Hkv = p.num_kv_heads, Hq = p.num_heads, G = Hq / Hkv;
    const int s = blockIdx.x / Hkv, h = blockIdx.x % Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    int npieces, c0 = 0, F = 0, R = 1;
    if (p.mode == kModeBalanced) {
        const int32_t *pre = p.ws_prefix;
        const int nt = pre[s + 1] - pre[s];
        if (nt == 0)
            return;
        const int total = Hkv * pre[p.num_seqs];
        R = max((total + p.grid - 1) / p.grid, p.min_tiles);
        F = Hkv * pre[s] + h * nt;
        c0 = F / R;
        const int c1 = (F + nt - 1) / R;
        if (c0 == c1)
            return;
        npieces = c1 - c0 + 1;
    } else {
        int L = __ldg(p.seq_lens + s);
        L = max(0, min(L, p.max_blocks * kBlockSize));
        const int nt = (L + kBlockSize - 1) / kBlockSize;
        npieces = (nt + p.part_tiles - 1) / p.part_tiles;
        if (npieces <= 1)
            return;
    }
    // partial row of piece pi, head g (same numbering the decode wrote)
    auto row = [&](int pi, int g) -> size_t {
        if (p.mode == kModeBalanced) {
            const int c = c0 + pi;
            const int slot = (c == c0 && F != c0 * R) ? 2 * c + 1 : 2 * c;
            return (size_t)slot * G + g;
        }
        return ((size_t)s * Hq + h * G + g) * p.p_max + pi;
    };

    for (int g = warp; g < G; g += 4) {
        float Mx = -INFINITY;
        for (int pi = lane; pi < npieces; pi += 32)
            Mx = fmaxf(Mx, p.ws_m[row(pi, g)]);
#pragma unroll
        for (int off = 16; off; off >>= 1)
            Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, off));
        float Wt = 0.f;
        for (int pi = lane; pi < npieces; pi += 32) {
            const size_t rw = row(pi, g);
            Wt += p.ws_l[rw] * exp2f((p.ws_m[rw] - Mx) * kLog2e);
        }
#pragma unroll
        for (int off = 16; off; off >>= 1)
            Wt += __shfl_xor_sync(0xffffffffu, Wt, off);
        if (lane == 0) {
            sM[g] = Mx;
            sW[g] = Wt;
        }
    }
    __syncthreads();

    constexpr int PER = (8 * D + 127) / 128;
    float O[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k)
        O[k] = 0.f;
    for (int base = 0; base < npieces; base += CH) {
        const int cnt = min(CH, npieces - base);
        for (int e = tid; e < cnt * G; e += 128) {
            const int pi = e / G, g = e % G;
            const size_t rw = row(base + pi, g);
            wts[pi][g] = p.ws_l[rw] * exp2f((p.ws_m[rw] - sM[g]) * kLog2e);
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const int e = tid + k * 128;
            if (e < G * D) {
                const int g = e / D, d = e % D;
                float acc = O[k];
                for (int pi = 0; pi < cnt; ++pi)
                    acc += wts[pi][g] * p.ws_o[row(base + pi, g) * D + d];
                O[k] = acc;
            }
        }
        __syncthreads();
    }
    T *out = reinterpret_cast<T *>(p.out);
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int e = tid + k * 128;
        if (e < G * D) {
            const int g = e / D, d = e % D;
            out[((size_t)s * Hq + h * G + g) * D + d] = E::from_f(O[k] / sW[g]);
        }
    }
}

template <typename T, int D>
inline void fill_kernel_set(KernelSet *ks)
{
    constexpr int W = 4;
    constexpr int S = 2;
    ks->decode = reinterpret_cast<const void *>(&decode_mma_kernel<T, D, W, S>);
    ks->merge = reinterpret_cast<const void *>(&merge_kernel<T, D>);
    ks->warps = W;
    ks->stages = S;
    ks->smem_fixed = MmaLayout<D, W, S>::fixed;
}

template <typename T>
inline bool kernels_for(int head_dim, int group, KernelSet *ks)
{
    if (group < 1 || group > 8)
        return false;
    if (head_dim == 128) {
        fill_kernel_set<T, 128>(ks);
        return true;
    }
    if (head_dim == 64) {
        fill_kernel_set<T, 64>(ks);
        return true;
    }
    return false;
}

}  // namespace pa
