// pa_prefix.cu -- attention of a group's query columns over its shared
// prefix, every prefix tile read from memory once.
//
// Parallel samples of one prompt name the same prompt blocks in their block
// tables (block sharing, section 系统实现要点 of the vLLM reading notes; the
// page-sharing row of its OS-paging table).  For the prefix they share, the
// query columns of a group and kv head -- every (sample, query head of the kv
// head) pair, group_size * G of them -- attend over the same K/V tiles.
//
// A thread block takes up to kPrefixCols of those columns and a chunk of the
// prefix's tiles.  One producer warp streams each tile once by TMA into a
// ring of stages (two pool blocks, 32 keys, a stage), and every consumer warp
// (8 columns each) multiplies the staged tiles against its columns with the
// decode's tensor-core steps (mma.sync m16n8k16, online softmax in base 2).
// A consumer's steps on one stage form a dependency chain, so the block is
// sized to its columns (up to 8 consumer warps) and kept small in registers,
// and several blocks share an SM.  Each column's result over the chunk is a
// partial (m, l, normalised o) in the form the decode's partial output uses,
// and the merge of pa_decode_shared_prefix folds the chunks' partials with
// the sample's own suffix (split-K with the log-sum-exp rule, ICML tutorial
// notes, section "内核优化").  On the way, the kernel writes the suffix
// decode's lengths (each sequence's tokens past the prefix).
//
// Prefix tiles hold 16 valid tokens each (the prefix is a whole number of
// blocks), so no key is masked.  Every wait is bounded: one that gives up
// records PA_DEVERR_TIMEOUT, and the producer lets its copies in flight land
// (bounded) before the block exits.
#include <algorithm>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_device.cuh"
#include "pa_shared.h"
#include "pagedattn.h"

namespace pa {
namespace {

// Up to kPrefixCols / 8 consumer warps and a producer warp a block.
// Registers a thread: three blocks of six warps per SM put five warps on a
// sub-partition (16384 registers).
constexpr int kPrefixRegs = 96;

template <int D>
struct PrefixShape {
    static constexpr int NB = D / 64;                     // 64-column boxes per tile
    static constexpr int BOX = kBlockSize * 128;          // 16 rows x 128 B
    static constexpr int TILE = NB * BOX;                 // K (or V) of one tile
    // a stage holds two tiles (32 keys): K and V of the first, then of the second
    static constexpr int STAGE = 4 * TILE;
    static constexpr int NSTG = D == 128 ? 4 : 8;         // ring depth
    static constexpr int KS = D / 16;                     // QK k-steps; PV m-tiles
    // +1024: the base is aligned up to the swizzle atom; then full[NSTG],
    // empty[NSTG] and the abort flag
    static constexpr int SMEM = 1024 + NSTG * STAGE + 2 * NSTG * 8 + 16;
    static_assert(STAGE % 1024 == 0, "stages keep the swizzle atom");
};

// L2 policy for tiles that the other column blocks of the chunk read too
__device__ __forceinline__ uint64_t l2_evict_normal_policy_()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint32_t swz_(int row, int chunk)
{
    return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

template <typename T, int D>
__global__ void __maxnreg__(kPrefixRegs)
prefix_attn_kernel(const PrefixParams p, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv)
{
    using Sh = PrefixShape<D>;
    using M = Mma<T>;
    constexpr int NS = Sh::NSTG, KS = Sh::KS;
    constexpr uint32_t FULL = 0xffffffffu;

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t bar_addr = sbase + NS * Sh::STAGE;
    auto full_bar = [&](int s) { return bar_addr + 8u * s; };
    auto empty_bar = [&](int s) { return bar_addr + 8u * (NS + s); };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + NS * Sh::STAGE + 16 * NS);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Hkv = p.num_kv_heads, Hq = p.num_heads, G = Hq / Hkv;
    // work item: (chunk, group and kv head, column block), column block fastest
    // so that the blocks sharing a chunk's tiles run side by side
    const int npairs = p.num_groups * Hkv;
    int b = blockIdx.x;
    const int cb = b % p.col_blocks;
    b /= p.col_blocks;
    const int pair = b % npairs, kc = b / npairs;
    const int g = pair / Hkv, h = pair - g * Hkv;
    const int t0 = kc * p.chunk_tiles;
    const int n = min(p.prefix_tiles, t0 + p.chunk_tiles) - t0;   // tiles of the chunk (>= 1)
    const int nsteps = (n + 1) / 2;                                // stages of two tiles
    const int c_lo = cb * kPrefixCols;
    const int ncols = min(kPrefixCols, p.cols - c_lo);            // columns of this block
    const int nw = (ncols + 7) / 8;                                // consumer warps at work
    const int pw = blockDim.x / 32 - 1;                            // the producer warp

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), nw);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();
    // a programmatic dependent launch: q and the tables may come from the
    // kernel before this one, so no thread reads them before it completes
    grid_dependents_launch();
    grid_dependency_wait();
    // the suffix decode's lengths: the tokens of each sequence past the prefix
    for (int s = blockIdx.x * blockDim.x + tid; s < p.num_seqs; s += gridDim.x * blockDim.x) {
        int L = __ldg(p.seq_lens + s) - p.prefix_tiles * kBlockSize;
        if (L < 0) {                                 // shorter than the shared prefix
            record_error(p.err, PA_DEVERR_SEQLEN_RANGE);
            L = 0;
        }
        p.lens_v[s] = L;
    }

    if (warp == pw) {
        // ---------------- producer: the chunk's tiles into the ring ----------
        const uint64_t pol = p.col_blocks > 1 ? l2_evict_normal_policy_() : l2_evict_first_policy();
        const int32_t *table = p.block_tables + (size_t)g * p.group_size * p.max_blocks + t0;
        auto fetch = [&](int i0) { return i0 + lane < n ? __ldg(table + i0 + lane) : 0; };
        int cur = fetch(0), nxt = fetch(32);
        int issued = 0;
        for (int i = 0; i < nsteps; ++i) {
            const int t = 2 * i;                                   // the stage's first tile
            if (t > 0 && (t & 31) == 0) {
                cur = nxt;
                nxt = fetch(t + 32);
            }
            const bool two = t + 1 < n;
            int phys[2] = {__shfl_sync(FULL, cur, t & 31), __shfl_sync(FULL, cur, (t + 1) & 31)};
            const int st = i % NS;
            bool ok = true;
            if (lane == 0)
                ok = !*abort_flag && (i < NS || mbar_wait_bounded(empty_bar(st), ((i / NS) - 1) & 1));
            if (!__shfl_sync(FULL, ok, 0)) {
                if (lane == 0 && !*abort_flag) {
                    *abort_flag = 1;
                    record_error(p.err, PA_DEVERR_TIMEOUT);
                }
                break;
            }
            if (lane == 0) {
                const uint32_t dst = sbase + st * Sh::STAGE;
                mbar_arrive_expect_tx(full_bar(st), (uint32_t)((two ? 4 : 2) * Sh::TILE));
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (u == 1 && !two)
                        break;
                    if ((unsigned)phys[u] >= (unsigned)p.num_blocks) {
                        record_error(p.err, PA_DEVERR_TABLE_RANGE);
                        phys[u] = 0;
                    }
                    const int row = (phys[u] * Hkv + h) * kBlockSize;
                    const uint32_t kd = dst + u * 2 * Sh::TILE;
#pragma unroll
                    for (int bx = 0; bx < Sh::NB; ++bx) {
                        tma_load_2d(kd + bx * Sh::BOX, &tmk, 64 * bx, row, full_bar(st), pol);
                        tma_load_2d(kd + Sh::TILE + bx * Sh::BOX, &tmv, 64 * bx, row, full_bar(st), pol);
                    }
                }
            }
            issued = i + 1;
        }
        // every copy issued lands before the block may exit (the last NS of
        // them are the ones a consumer may not have waited for)
        if (lane == 0)
            for (int x = issued > NS ? issued - NS : 0; x < issued; ++x)
                mbar_wait_bounded(full_bar(x % NS), (uint32_t)((x / NS) & 1));
        return;
    }
    if (warp >= nw)
        return;
    // ---------------- consumer warp: 8 query columns ----------------
    // Lane geometry of the decode: in S[16 tokens x 8 columns] and in
    // O^T[head_dim x 8 columns] a lane owns columns 2qd and 2qd + 1, rows r
    // and r + 8; B column r of Q^T is its to load.
    const int r = lane >> 2, qd = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;                  // ldmatrix: matrix, row
    const int krow = ((mi & 1) << 3) + rr, kcs = mi >> 1;     // K (A operand, row-major)
    const int vrow = ((mi >> 1) << 3) + rr, vcs = mi & 1;     // V (A operand via .trans)
    const int cw = c_lo + warp * 8;                           // this warp's first column

    // Q^T fragments: column c = (sample c / G, query head h G + c % G)
    uint32_t qf[KS][2];
    {
        const int c = cw + r;
        const bool valid = c < p.cols;
        const int smp = valid ? c / G : 0, hq = h * G + (valid ? c % G : 0);
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
            static_cast<const T *>(p.q) + ((size_t)(g * p.group_size + smp) * Hq + hq) * D);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qf[ks][0] = valid ? __ldg(qrow + (16 * ks + 2 * qd) / 2) : 0u;
            qf[ks][1] = valid ? __ldg(qrow + (16 * ks + 8 + 2 * qd) / 2) : 0u;
        }
    }
    float o[KS][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c)
            o[mt][c] = 0.f;

    for (int i = 0; i < nsteps; ++i) {
        const int st = i % NS;
        const bool two = 2 * i + 1 < n;                           // the stage's second tile
        if (!__all_sync(FULL, !*abort_flag && mbar_wait_bounded(full_bar(st), (i / NS) & 1))) {
            if (lane == 0 && !*abort_flag) {
                *abort_flag = 1;
                record_error(p.err, PA_DEVERR_TIMEOUT);
            }
            return;                                   // no partial: the call has failed
        }
        const uint32_t ka = sbase + st * Sh::STAGE, va = ka + Sh::TILE;
        const uint32_t kb = va + Sh::TILE, vb = kb + Sh::TILE;
        // S = K . Q^T for both tiles, one accumulator each (two chains)
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t a[4];
            const uint32_t off = (ks >> 2) * Sh::BOX + swz_(krow, 2 * (ks & 3) + kcs);
            ldsm_x4(ka + off, a[0], a[1], a[2], a[3]);
            M::run(sa, a, qf[ks][0], qf[ks][1]);
            if (two) {
                ldsm_x4(kb + off, a[0], a[1], a[2], a[3]);
                M::run(sb, a, qf[ks][0], qf[ks][1]);
            }
        }
        // scores: tile a tokens r, r+8; tile b the same (-inf without it)
        const float x0 = sa[0] * p.scale_log2, x1 = sa[1] * p.scale_log2;
        const float x2 = sa[2] * p.scale_log2, x3 = sa[3] * p.scale_log2;
        const float y0 = two ? sb[0] * p.scale_log2 : -INFINITY;
        const float y1 = two ? sb[1] * p.scale_log2 : -INFINITY;
        const float y2 = two ? sb[2] * p.scale_log2 : -INFINITY;
        const float y3 = two ? sb[3] * p.scale_log2 : -INFINITY;
        float mx0 = fmaxf(fmaxf(x0, x2), fmaxf(y0, y2)), mx1 = fmaxf(fmaxf(x1, x3), fmaxf(y1, y3));
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
        const float q0 = exp2f(y0 - m0), q1 = exp2f(y1 - m1);
        const float q2 = exp2f(y2 - m0), q3 = exp2f(y3 - m1);
        l0 += (p0 + p2) + (q0 + q2);
        l1 += (p1 + p3) + (q1 + q3);
        // P^T as the B operand: the tokens become columns
        const uint32_t pa0 = movmatrix_trans(M::pack(p0, p1));
        const uint32_t pa1 = movmatrix_trans(M::pack(p2, p3));
        const uint32_t pb0 = movmatrix_trans(M::pack(q0, q1));
        const uint32_t pb1 = movmatrix_trans(M::pack(q2, q3));
        // O^T += V^T . P^T, tile by tile (a missing second tile's stage holds
        // stale rows: its products are skipped, not weighted by zero)
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            uint32_t a[4];
            const uint32_t off = (mt >> 2) * Sh::BOX + swz_(vrow, 2 * (mt & 3) + vcs);
            ldsm_x4_trans(va + off, a[0], a[1], a[2], a[3]);
            M::run(o[mt], a, pa0, pa1);
            if (two) {
                ldsm_x4_trans(vb + off, a[0], a[1], a[2], a[3]);
                M::run(o[mt], a, pb0, pb1);
            }
        }
        // the stage is free once every lane has read it
        __syncwarp();
        if (lane == 0)
            mbar_arrive(empty_bar(st));
    }

    // ---- the columns' partials over the chunk: m (natural log), l, o / l ----
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(FULL, l0, off);
        l1 += __shfl_xor_sync(FULL, l1, off);
    }
    const float inv0 = 1.f / l0, inv1 = 1.f / l1;
    const int c0 = cw + 2 * qd, c1 = c0 + 1;
    const size_t row0 = ((size_t)kc * npairs + pair) * p.cols + c0, row1 = row0 + 1;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
        const int d0 = 16 * mt + r;
        if (c0 < p.cols) {
            p.xo[row0 * D + d0] = o[mt][0] * inv0;
            p.xo[row0 * D + d0 + 8] = o[mt][2] * inv0;
        }
        if (c1 < p.cols) {
            p.xo[row1 * D + d0] = o[mt][1] * inv1;
            p.xo[row1 * D + d0 + 8] = o[mt][3] * inv1;
        }
    }
    if (r == 0) {
        if (c0 < p.cols) {
            p.xm[row0] = m0 * kLn2;
            p.xl[row0] = l0;
        }
        if (c1 < p.cols) {
            p.xm[row1] = m1 * kLn2;
            p.xl[row1] = l1;
        }
    }
}

}  // namespace

PrefixKernel prefix_kernel(const PrefixParams &p, bool bf16, int head_dim)
{
    PrefixKernel k{};
    if (head_dim == 128) {
        k.fn = bf16 ? reinterpret_cast<const void *>(&prefix_attn_kernel<__nv_bfloat16, 128>)
                    : reinterpret_cast<const void *>(&prefix_attn_kernel<__half, 128>);
        k.smem = PrefixShape<128>::SMEM;
    } else {
        k.fn = bf16 ? reinterpret_cast<const void *>(&prefix_attn_kernel<__nv_bfloat16, 64>)
                    : reinterpret_cast<const void *>(&prefix_attn_kernel<__half, 64>);
        k.smem = PrefixShape<64>::SMEM;
    }
    // consumer warps for the widest column block, and the producer
    k.threads = 32 * ((std::min(p.cols, kPrefixCols) + 7) / 8 + 1);
    k.blocks = p.nchunks * p.num_groups * p.num_kv_heads * p.col_blocks;
    return k;
}

}  // namespace pa
