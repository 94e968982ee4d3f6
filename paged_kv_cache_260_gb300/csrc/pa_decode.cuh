// pa_decode.cuh -- paged decode attention for sm_103a.
//
// What it computes: for each sequence s and query head h,
//     out[s][h] = sum_t softmax_t(scale * q[s][h] . k_t) v_t ,  t < seq_len(s)
// with k_t, v_t read through the sequence's block table (attention over a
// KV cache kept in 16-token blocks that are not contiguous in memory; the
// block-table figure of "PagedAttention：vLLM 系统论文", section 核心思想).
// The score row is never stored: a running max and running sum rescale the
// partial result as tiles arrive (online softmax, vLLM deep notes, section
// "核心思想：Tiling + Online Softmax").  Long runs are split along the sequence
// and the pieces merged with the log-sum-exp rule (FlashDecoding split-K, ICML
// tutorial notes, section "内核优化").
//
// How it maps onto GB300:
//  * Unit of data: one (physical block, kv head) tile = 16 tokens x head_dim,
//    contiguous in the pool (4 KiB of K + 4 KiB of V at head_dim 128).  Each
//    tile is fetched with two 1-D bulk copies (TMA) into shared memory and
//    completes on an mbarrier; nothing else touches HBM on the hot path.
//  * A persistent grid (SMs x resident blocks) walks a flat list of tiles
//    ordered (sequence, kv head, block).  Balanced mode gives every thread
//    block the same number of tiles; fixed mode hands out whole partitions;
//    whole mode hands out whole (sequence, kv head) runs.
//  * Within a thread block each warp owns its own ring of copy stages and
//    takes every W-th tile of the block's current run; warps meet only at
//    the end of a run to combine their softmax states in shared memory.
//  * One warp serves the whole query group (G heads) of a kv head, so each
//    K/V byte is read from HBM once per decode.  Lanes split the tile as
//    (half: 8 tokens) x (16 lanes: head_dim/16 channels); per-token dot
//    products are finished by a butterfly reduce-scatter of the G x tokens
//    partial sums across the 16 lanes of a half, which also hands each lane
//    the scores it applies the softmax to.  Packed fp32x2 FMAs do the math.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

template <int D, int G>
struct Shape {
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(G >= 1 && G <= 8, "group");
    static constexpr int DL = D / 16;                                       // channels per lane
    static constexpr int GP = G == 1 ? 1 : G == 2 ? 2 : G <= 4 ? 4 : 8;     // padded group
    static constexpr int TR = G <= 4 ? 8 : 4;                               // tokens per half per round
    static constexpr int NR = 8 / TR;                                       // rounds per tile
    static constexpr int VPH = TR * GP;                                     // partial sums per half
    static constexpr int NF = VPH >= 16 ? VPH / 16 : 1;                     // scores kept per lane
    static constexpr int LPH = VPH >= 16 ? TR / NF : 16;                    // lanes per head in a half
    static constexpr int TILE = kBlockSize * D * 2;                         // bytes of K (or V) per tile
    static constexpr int QB = G * D * 2;                                    // bytes of the q group
    static constexpr int QSLOT = (QB + 127) / 128 * 128;
    static constexpr int STAGE = 2 * TILE + QSLOT;
};

template <int D, int G, int W, int S>
struct Layout {
    using Sh = Shape<D, G>;
    static constexpr size_t stages = (size_t)W * S * Sh::STAGE;
    static constexpr size_t pbuf = (size_t)W * 16 * Sh::GP * 4;
    static constexpr size_t cm = (size_t)W * Sh::GP * 4;
    static constexpr size_t cl = cm;
    static constexpr size_t cacc = (size_t)W * G * D * 4;
    static constexpr size_t bars = (size_t)W * S * 8;
    static constexpr size_t fixed = stages + pbuf + cm + cl + cacc + bars;
};

// ---------------------------------------------------------------------------
// Work walker: enumerates the runs ("pieces") one thread block processes.  A
// piece is a range [tb, te) of tiles of the (sequence s, kv head h) run.
// Every thread of the block evaluates it identically.
// ---------------------------------------------------------------------------
struct Walker {
    // constants
    const int32_t *pre;   // unit prefix [n + 1] (tiles, partitions or 0/1 per sequence)
    const int32_t *lens;  // clamped lengths [n]
    int n, hkv, mode, pt;
    // state
    int s, h, tb, te, nt;
    int cur;      // balanced: first flat tile of (s, h); fixed/whole: flat item index
    int end;      // balanced: end of the block's tile range; fixed/whole: end item
    int part;     // fixed: partition index within (s, h)
    int np;       // fixed/whole: partitions of sequence s
    bool valid;
    bool first;   // first piece of this thread block

    __device__ __forceinline__ int find_seq(int x) const
    {
        // largest s with hkv * pre[s] <= x (sequences without units are skipped)
        int lo = 0, hi = n - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (hkv * pre[mid] <= x)
                lo = mid;
            else
                hi = mid - 1;
        }
        return lo;
    }

    __device__ __forceinline__ int tiles_of(int seq) const { return (lens[seq] + kBlockSize - 1) / kBlockSize; }

    __device__ __forceinline__ void set_fixed_piece()
    {
        nt = tiles_of(s);
        if (mode == kModeFixed) {
            tb = part * pt;
            te = min(nt, tb + pt);
        } else {
            tb = 0;
            te = nt;
        }
    }

    __device__ __forceinline__ void init(const int32_t *pre_, const int32_t *lens_, int n_, int hkv_,
                                         int mode_, int pt_, int min_tiles, int grid, int bid)
    {
        pre = pre_;
        lens = lens_;
        n = n_;
        hkv = hkv_;
        mode = mode_;
        pt = pt_;
        first = true;
        const int total = hkv * pre[n];
        if (mode == kModeBalanced) {
            int R = (total + grid - 1) / grid;
            R = max(R, min_tiles);
            const long long a = (long long)bid * R;
            valid = a < total;
            if (!valid)
                return;
            const int A = (int)a;
            end = min(total, A + R);
            s = find_seq(A);
            nt = pre[s + 1] - pre[s];
            const int rel = A - hkv * pre[s];
            h = rel / nt;
            cur = hkv * pre[s] + h * nt;
            tb = A - cur;
            te = min(nt, end - cur);
        } else {
            const int i0 = (int)((long long)bid * total / grid);
            end = (int)((long long)(bid + 1) * total / grid);
            valid = i0 < end;
            if (!valid)
                return;
            cur = i0;
            s = find_seq(i0);
            np = pre[s + 1] - pre[s];
            const int rel = i0 - hkv * pre[s];
            h = rel / np;
            part = rel % np;
            set_fixed_piece();
        }
    }

    __device__ __forceinline__ void next_seq()
    {
        do {
            ++s;
        } while (s < n && pre[s + 1] == pre[s]);
    }

    __device__ __forceinline__ void next()
    {
        first = false;
        if (mode == kModeBalanced) {
            cur += nt;
            if (cur >= end) {
                valid = false;
                return;
            }
            if (++h == hkv) {
                h = 0;
                next_seq();
                nt = pre[s + 1] - pre[s];
            }
            tb = 0;
            te = min(nt, end - cur);
        } else {
            if (++cur >= end) {
                valid = false;
                return;
            }
            if (++part == np) {
                part = 0;
                if (++h == hkv) {
                    h = 0;
                    next_seq();
                    np = pre[s + 1] - pre[s];
                }
            }
            set_fixed_piece();
        }
    }

    __device__ __forceinline__ bool whole() const
    {
        return mode == kModeBalanced ? (tb == 0 && te == nt) : (mode == kModeWhole || np == 1);
    }
};

// Units a sequence of (clamped) length L contributes to the flat work list.
__device__ __forceinline__ int seq_units(int L, int mode, int pt)
{
    const int nt = (L + kBlockSize - 1) / kBlockSize;
    if (mode == kModeBalanced)
        return nt;
    if (mode == kModeFixed)
        return (nt + pt - 1) / pt;
    return nt > 0 ? 1 : 0;
}

// Clamp the lengths into shared memory and build the exclusive unit prefix.
template <int W>
__device__ __forceinline__ void build_prefix(const DecodeParams &p, int32_t *pre, int32_t *lens)
{
    __shared__ int warp_sum[W];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = p.num_seqs;
    const int nthr = W * 32;
    const int per = (n + nthr - 1) / nthr;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    const int maxlen = p.max_blocks * kBlockSize;
    int sum = 0;
    bool bad = false;
    for (int s = lo; s < hi; ++s) {
        int L = __ldg(p.seq_lens + s);
        if (L < 0 || L > maxlen) {
            bad = true;
            L = L < 0 ? 0 : maxlen;
        }
        lens[s] = L;
        sum += seq_units(L, p.mode, p.part_tiles);
    }
    if (bad && blockIdx.x == 0)
        record_error(p.err, PA_DEVERR_SEQLEN_RANGE);
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        warp_sum[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w)
        before += warp_sum[w];
    int run = before + incl - sum;
    for (int s = lo; s < hi; ++s) {
        pre[s] = run;
        run += seq_units(lens[s], p.mode, p.part_tiles);
    }
    if (tid == nthr - 1)
        pre[n] = before + incl;
}

template <typename T, int D, int G, int W, int S>
__global__ void __launch_bounds__(W * 32) decode_kernel(const DecodeParams p)
{
    using Sh = Shape<D, G>;
    using Lay = Layout<D, G, W, S>;
    using E = Elem<T>;
    constexpr int DL = Sh::DL, GP = Sh::GP, TR = Sh::TR, NR = Sh::NR, VPH = Sh::VPH;
    constexpr int NF = Sh::NF, LPH = Sh::LPH, DL2 = DL / 2;
    constexpr uint32_t FULL = 0xffffffffu;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stage_base = smem;
    float *pbuf_all = reinterpret_cast<float *>(smem + Lay::stages);
    float *cm = pbuf_all + W * 16 * GP;
    float *cl = cm + W * GP;
    float *cacc = cl + W * GP;
    uint64_t *bars = reinterpret_cast<uint64_t *>(cacc + W * G * D);
    int32_t *pre = reinterpret_cast<int32_t *>(bars + W * S);
    int32_t *lens = pre + p.num_seqs + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hh = lane >> 4, j = lane & 15;
    const int n = p.num_seqs, Hkv = p.num_kv_heads, Hq = p.num_heads;

    if (lane == 0) {
        for (int st = 0; st < S; ++st)
            mbar_init(smem_addr(&bars[warp * S + st]), 1);
        mbar_init_fence();
    }
    build_prefix<W>(p, pre, lens);
    __syncthreads();

    // the merge of balanced mode needs the prefix; sequences without tokens
    // get zeros (no piece ever covers them)
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

    // ---- this warp's scores: value index v = g * TR + t of a half ----
    const int v0 = VPH >= 16 ? j * NF : (j >> 1);
    const int g_own = v0 / TR;
    const int t_own0 = v0 % TR;
    const bool counts = VPH >= 16 || (j & 1) == 0;  // duplicated lanes count once

    const uint64_t pol = l2_evict_first_policy();
    const uint32_t bar0 = smem_addr(&bars[warp * S]);
    unsigned char *wst = stage_base + (size_t)warp * S * Sh::STAGE;
    float *pbuf = pbuf_all + warp * 16 * GP;

    // ---- producer: issue this warp's tiles S ahead of the consumer ----
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
            const size_t tile_el = ((size_t)phys * Hkv + prod.h) * (kBlockSize * D);
            const uint32_t bar = bar0 + st * 8;
            const uint32_t dst = smem_addr(wst + (size_t)st * Sh::STAGE);
            mbar_arrive_expect_tx(bar, 2 * Sh::TILE + (pfirst ? Sh::QB : 0));
            bulk_load(dst, reinterpret_cast<const T *>(p.k_cache) + tile_el, Sh::TILE, bar, pol);
            bulk_load(dst + Sh::TILE, reinterpret_cast<const T *>(p.v_cache) + tile_el, Sh::TILE, bar, pol);
            if (pfirst)
                bulk_load(dst + 2 * Sh::TILE,
                          reinterpret_cast<const T *>(p.q) + ((size_t)prod.s * Hq + prod.h * G) * D,
                          Sh::QB, bar);
        }
        pfirst = false;
        ptile += W;
        advance();
        if (!pdone && lane == 0)
            pphys = __ldg(p.block_tables + (size_t)prod.s * p.max_blocks + ptile);
        ++issued;
    };
    for (int st = 0; st < S; ++st)
        produce(st);

    // ---- consumer ----
    float2 q2[G][DL2];
    float2 acc[G][DL2];
    float m_own, l_own;
    int it = 0;
    bool aborted = false;
    int abort_it = 0;

    while (cons.valid) {
        m_own = -INFINITY;
        l_own = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int c = 0; c < DL2; ++c)
                acc[g][c] = make_float2(0.f, 0.f);
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
            const unsigned char *sb = wst + (size_t)st * Sh::STAGE;
            const T *Kt = reinterpret_cast<const T *>(sb);
            const T *Vt = reinterpret_cast<const T *>(sb + Sh::TILE);
            if (need_q) {
                const T *Qs = reinterpret_cast<const T *>(sb + 2 * Sh::TILE);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const uint32_t *src = reinterpret_cast<const uint32_t *>(Qs + g * D + j * DL);
#pragma unroll
                    for (int c = 0; c < DL2; ++c) {
                        float2 f = E::to_f2(src[c]);
                        q2[g][c] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
                    }
                }
                need_q = false;
            }
            const int nvalid = min(kBlockSize, L - tile * kBlockSize);

#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r * TR >= nvalid)
                    break;  // every token of this round is past the end
                // -- partial dot products over this lane's channels --
                float part[VPH];
#pragma unroll
                for (int v = 0; v < VPH; ++v)
                    part[v] = 0.f;
#pragma unroll
                for (int t = 0; t < TR; ++t) {
                    const int tt = hh * 8 + r * TR + t;
                    float2 kf[DL2];
                    if constexpr (DL == 8) {
                        const uint4 raw = *reinterpret_cast<const uint4 *>(Kt + tt * D + j * DL);
                        kf[0] = E::to_f2(raw.x);
                        kf[1] = E::to_f2(raw.y);
                        kf[2] = E::to_f2(raw.z);
                        kf[3] = E::to_f2(raw.w);
                    } else {
                        const uint2 raw = *reinterpret_cast<const uint2 *>(Kt + tt * D + j * DL);
                        kf[0] = E::to_f2(raw.x);
                        kf[1] = E::to_f2(raw.y);
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float2 a = __fmul2_rn(q2[g][0], kf[0]);
#pragma unroll
                        for (int c = 1; c < DL2; ++c)
                            a = __ffma2_rn(q2[g][c], kf[c], a);
                        part[g * TR + t] = a.x + a.y;
                    }
                }
                // -- butterfly reduce-scatter across the 16 lanes of the half --
                {
                    int cnt = VPH;
#pragma unroll
                    for (int m = 8; m >= 1; m >>= 1) {
                        if (cnt >= 2) {
                            const int half = cnt / 2;
                            const bool upper = (j & m) != 0;
#pragma unroll
                            for (int i = 0; i < half; ++i) {
                                const float send = upper ? part[i] : part[half + i];
                                const float keep = upper ? part[half + i] : part[i];
                                part[i] = keep + __shfl_xor_sync(FULL, send, m);
                            }
                            cnt = half;
                        } else {
                            part[0] += __shfl_xor_sync(FULL, part[0], m);
                        }
                    }
                }
                // -- scores of this lane: part[0..NF) --
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < NF; ++i) {
                    const int tt = hh * 8 + r * TR + t_own0 + i;
                    if (tt >= nvalid)
                        part[i] = -INFINITY;
                    mx = fmaxf(mx, part[i]);
                }
#pragma unroll
                for (int o = 1; o < LPH; o <<= 1)
                    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
                mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 16));
                if (__any_sync(FULL, mx > m_own)) {
                    const float m_new = fmaxf(m_own, mx);
                    const float alpha = exp2f(m_own - m_new);
                    m_own = m_new;
                    l_own *= alpha;
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float a = __shfl_sync(FULL, alpha, g * LPH);
                        const float2 a2 = make_float2(a, a);
#pragma unroll
                        for (int c = 0; c < DL2; ++c)
                            acc[g][c] = __fmul2_rn(acc[g][c], a2);
                    }
                }
#pragma unroll
                for (int i = 0; i < NF; ++i) {
                    const float pv = exp2f(part[i] - m_own);
                    if (counts)
                        l_own += pv;
                    if (g_own < G)
                        pbuf[(hh * 8 + r * TR + t_own0 + i) * GP + g_own] = pv;
                }
                __syncwarp();
                // -- weighted sum of values --
#pragma unroll
                for (int t = 0; t < TR; ++t) {
                    const int tt = hh * 8 + r * TR + t;
                    float2 vf[DL2];
                    if constexpr (DL == 8) {
                        const uint4 raw = *reinterpret_cast<const uint4 *>(Vt + tt * D + j * DL);
                        vf[0] = E::to_f2(raw.x);
                        vf[1] = E::to_f2(raw.y);
                        vf[2] = E::to_f2(raw.z);
                        vf[3] = E::to_f2(raw.w);
                    } else {
                        const uint2 raw = *reinterpret_cast<const uint2 *>(Vt + tt * D + j * DL);
                        vf[0] = E::to_f2(raw.x);
                        vf[1] = E::to_f2(raw.y);
                    }
                    if (tt >= nvalid) {
                        // slots past the end may hold anything, NaN included
#pragma unroll
                        for (int c = 0; c < DL2; ++c)
                            vf[c] = make_float2(0.f, 0.f);
                    }
                    float pg[GP];
                    if constexpr (GP >= 4) {
#pragma unroll
                        for (int g4 = 0; g4 < GP; g4 += 4) {
                            const float4 x = *reinterpret_cast<const float4 *>(pbuf + tt * GP + g4);
                            pg[g4] = x.x;
                            pg[g4 + 1] = x.y;
                            pg[g4 + 2] = x.z;
                            pg[g4 + 3] = x.w;
                        }
                    } else if constexpr (GP == 2) {
                        const float2 x = *reinterpret_cast<const float2 *>(pbuf + tt * GP);
                        pg[0] = x.x;
                        pg[1] = x.y;
                    } else {
                        pg[0] = pbuf[tt];
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float2 pp = make_float2(pg[g], pg[g]);
#pragma unroll
                        for (int c = 0; c < DL2; ++c)
                            acc[g][c] = __ffma2_rn(pp, vf[c], acc[g][c]);
                    }
                }
                __syncwarp();
            }
            if (!aborted)
                produce(st);
            ++it;
        }

        // ---- end of piece: combine the warps' states ----
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int c = 0; c < DL2; ++c) {
                acc[g][c].x += __shfl_xor_sync(FULL, acc[g][c].x, 16);
                acc[g][c].y += __shfl_xor_sync(FULL, acc[g][c].y, 16);
            }
        float lt = l_own;
#pragma unroll
        for (int o = 1; o < LPH; o <<= 1)
            lt += __shfl_xor_sync(FULL, lt, o);
        lt += __shfl_xor_sync(FULL, lt, 16);
        if (hh == 0) {
            if ((j % LPH) == 0 && g_own < G) {
                cm[warp * GP + g_own] = m_own;
                cl[warp * GP + g_own] = lt;
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float *dst = cacc + (warp * G + g) * D + j * DL;
#pragma unroll
                for (int c = 0; c < DL2; ++c)
                    reinterpret_cast<float2 *>(dst)[c] = acc[g][c];
            }
        }
        __syncthreads();
        {
            const bool whole = cons.whole();
            for (int e = tid; e < G * D; e += W * 32) {
                const int g = e / D, d = e % D;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < W; ++w)
                    M = fmaxf(M, cm[w * GP + g]);
                float Ls = 0.f, O = 0.f;
#pragma unroll
                for (int w = 0; w < W; ++w) {
                    const float mw = cm[w * GP + g];
                    const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
                    Ls += f * cl[w * GP + g];
                    O += f * cacc[(w * G + g) * D + d];
                }
                const float res = O / Ls;
                if (whole) {
                    T *o = reinterpret_cast<T *>(p.out);
                    o[((size_t)cons.s * Hq + cons.h * G + g) * D + d] = E::from_f(res);
                } else {
                    size_t row;
                    if (p.mode == kModeBalanced)
                        row = (size_t)(2 * blockIdx.x + (cons.first ? 0 : 1)) * G + g;
                    else
                        row = ((size_t)cons.s * Hq + cons.h * G + g) * p.p_max + cons.part;
                    p.ws_o[row * D + d] = res;
                    if (d == 0) {
                        p.ws_m[row] = M * kLn2;
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
// Log-sum-exp merge of split runs: M = max m_p, w_p = l_p exp(m_p - M),
// out = sum_p w_p o_p / sum_p w_p.  One thread block per (sequence, kv head).
// ---------------------------------------------------------------------------
template <typename T, int D, int G>
__global__ void __launch_bounds__(128) merge_kernel(const DecodeParams p)
{
    using E = Elem<T>;
    constexpr int CH = 64;  // pieces whose weights are staged at a time
    __shared__ float sM[G], sW[G];
    __shared__ float wts[CH][G];
    const int Hkv = p.num_kv_heads, Hq = p.num_heads;
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
    auto row = [&](int pi, int g) -> size_t {
        if (p.mode == kModeBalanced) {
            const int c = c0 + pi;
            const int slot = (c == c0 && F != c0 * R) ? 2 * c + 1 : 2 * c;
            return (size_t)slot * G + g;
        }
        return ((size_t)s * Hq + h * G + g) * p.p_max + pi;
    };

    for (int g = warp; g < G; g += 4) {
        float M = -INFINITY;
        for (int pi = lane; pi < npieces; pi += 32)
            M = fmaxf(M, p.ws_m[row(pi, g)]);
#pragma unroll
        for (int o = 16; o; o >>= 1)
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float Wt = 0.f;
        for (int pi = lane; pi < npieces; pi += 32) {
            const size_t r = row(pi, g);
            Wt += p.ws_l[r] * exp2f((p.ws_m[r] - M) * kLog2e);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1)
            Wt += __shfl_xor_sync(0xffffffffu, Wt, o);
        if (lane == 0) {
            sM[g] = M;
            sW[g] = Wt;
        }
    }
    __syncthreads();

    constexpr int PER = (G * D + 127) / 128;
    float O[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k)
        O[k] = 0.f;
    for (int base = 0; base < npieces; base += CH) {
        const int cnt = min(CH, npieces - base);
        for (int e = tid; e < cnt * G; e += 128) {
            const int pi = e / G, g = e % G;
            const size_t r = row(base + pi, g);
            wts[pi][g] = p.ws_l[r] * exp2f((p.ws_m[r] - sM[g]) * kLog2e);
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

template <typename T, int D, int G>
inline void fill_kernel_set(KernelSet *ks)
{
    constexpr int W = 4;
    constexpr int S = 2;
    ks->decode = reinterpret_cast<const void *>(&decode_kernel<T, D, G, W, S>);
    ks->merge = reinterpret_cast<const void *>(&merge_kernel<T, D, G>);
    ks->warps = W;
    ks->stages = S;
    ks->smem_fixed = Layout<D, G, W, S>::fixed;
}

template <typename T>
inline bool kernels_for(int head_dim, int group, KernelSet *ks)
{
#define PA_CASE(DD, GG)                        \
    if (head_dim == DD && group == GG) {       \
        fill_kernel_set<T, DD, GG>(ks);        \
        return true;                           \
    }
    PA_CASE(128, 1) PA_CASE(128, 2) PA_CASE(128, 3) PA_CASE(128, 4)
    PA_CASE(128, 5) PA_CASE(128, 6) PA_CASE(128, 7) PA_CASE(128, 8)
    PA_CASE(64, 1) PA_CASE(64, 2) PA_CASE(64, 3) PA_CASE(64, 4)
    PA_CASE(64, 5) PA_CASE(64, 6) PA_CASE(64, 7) PA_CASE(64, 8)
#undef PA_CASE
    return false;
}

}  // namespace pa
