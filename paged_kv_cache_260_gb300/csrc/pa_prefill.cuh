// pa_prefill.cuh -- paged chunked-prefill attention on the fifth-generation
// tensor cores (tcgen05).
//
// The chunk of c new tokens of a sequence of length L (their K/V already in
// the pool) attends causally over the pool: the token at position
// p = L - c + i sees positions [0, p].  Chunked prefill: vLLM deep notes,
// section "调度优化：Continuous / Chunked / Disaggregated"; forum summary,
// section "Sarathi-Serve：Chunked-Prefill技术".  K/V are reached through the
// block table of "PagedAttention：vLLM 系统论文", section 核心思想.
//
// One thread block computes 128 rows = (token, q head) pairs of one sequence
// and one kv head: 128 / G consecutive chunk tokens times the G q heads that
// share the kv head, so every K/V tile it stages serves all of them.
// Warp roles (192 threads):
//   warp 0    one lane: TMA producer of K and V tiles of 64 keys (4 pool
//             blocks x 16 rows x 128-byte boxes) into a ring of 3 slots;
//   warp 1    TMEM owner; one lane issues the MMAs:
//               S_j = Q . K_j^T            (M 128, N 64, K = head_dim)
//               O  += P_j . V_j            (M 128, N head_dim, K 64)
//             S is double-buffered in TMEM so S_{j+1} runs while the
//             softmax warps work on S_j;
//   warps 2-5 one thread per row (its TMEM lane): scores from TMEM, causal
//             mask, online softmax in base 2 with a lazy rescale of O (only
//             when the running maximum grows by more than 2^8), P written to
//             shared memory as the A operand of the next MMA, and the final
//             O / l written out.
// TMEM: columns [0, 128) hold the two S buffers, [128, 128 + head_dim) O.
// Every wait is bounded; a wait that gives up records PA_DEVERR_TIMEOUT and
// the block drains its copies and MMAs before it frees TMEM and exits.
#pragma once

#include <cuda.h>
#include <type_traits>

#include "pa_device.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

template <int D>
struct PrefillShape {
    static constexpr int BM = kPrefillRows;                 // rows per block
    static constexpr int BN = 64;                           // keys per tile
    static constexpr int NSLOT = 3;                         // K/V ring
    static constexpr int HALVES = D / 64;                   // 128-byte column boxes
    static constexpr int BOX = 2048;                        // 16 rows x 128 B
    static constexpr int Q_BYTES = BM * D * 2;              // [half][128 rows][128 B]
    static constexpr int SLOT_BYTES = BN * D * 2;           // [half][4 blocks][16 rows][128 B]
    static constexpr int P_BYTES = BM * BN * 2;             // [128 rows][128 B]
    static constexpr int OFF_SLOT = Q_BYTES;
    static constexpr int OFF_P = OFF_SLOT + NSLOT * SLOT_BYTES;
    static constexpr int OFF_BAR = OFF_P + P_BYTES;
    static constexpr int NBAR = 11;                         // full[3] empty[3] s[2] p o drain
    static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;   // + alignment slack
    static constexpr int THREADS = 192;
    static constexpr uint32_t TMEM_COLS = 256;
    static constexpr uint32_t COL_S = 0;
    static constexpr uint32_t COL_O = 128;
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(OFF_P % 1024 == 0 && OFF_SLOT % 1024 == 0, "swizzle atoms");
};

template <typename T, int D>
__global__ void __launch_bounds__(192, 2)
prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv)
{
    using Sh = PrefillShape<D>;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t FULL = 0xffffffffu;

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t q_addr = sbase;
    const uint32_t slot_addr = sbase + Sh::OFF_SLOT;
    const uint32_t p_addr = sbase + Sh::OFF_P;
    const uint32_t bar_addr = sbase + Sh::OFF_BAR;
    // barrier addresses
    auto full_bar = [&](int s) { return bar_addr + 8u * s; };
    auto empty_bar = [&](int s) { return bar_addr + 8u * (3 + s); };
    auto s_bar = [&](int b) { return bar_addr + 8u * (6 + b); };
    const uint32_t p_bar = bar_addr + 8u * 8;
    const uint32_t o_bar = bar_addr + 8u * 9;
    const uint32_t drain_bar = bar_addr + 8u * 10;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Sh::OFF_BAR + Sh::NBAR * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Hkv = p.num_kv_heads, Hq = p.num_heads, G = Hq / Hkv;
    const int TPC = Sh::BM / G;                   // chunk tokens per block
    const int per_rank = p.num_seqs * Hkv;
    const int rank = blockIdx.x / per_rank;
    const int s = (blockIdx.x % per_rank) / Hkv;
    const int h = blockIdx.x % Hkv;

    // ---- the block's rows and key range (uniform over the block) ----------
    const int L = __ldg(p.seq_lens + s);
    const int qs = __ldg(p.query_start + s);
    const int c = __ldg(p.query_start + s + 1) - qs;
    if (L < 0 || L > p.max_blocks * kBlockSize) {
        if (rank == 0 && h == 0 && tid == 0)
            record_error(p.err, PA_DEVERR_SEQLEN_RANGE);
        return;
    }
    if (c < 0 || c > L) {
        if (rank == 0 && h == 0 && tid == 0)
            record_error(p.err, PA_DEVERR_QUERY_RANGE);
        return;
    }
    const int nq = (c + TPC - 1) / TPC;
    if (nq > p.q_ranks && rank == 0 && h == 0 && tid == 0)
        record_error(p.err, PA_DEVERR_QUERY_RANGE);   // max_query_len too small
    if (rank >= nq)
        return;
    const int tile = nq - 1 - rank;               // rank 0 = the last (longest) tile
    const int t0 = tile * TPC;
    const int t_end = min(t0 + TPC, c);
    const int p_last = L - c + t_end - 1;         // position of the block's last row
    const int nt = p_last / Sh::BN + 1;           // key tiles
    const int nblk = (L + kBlockSize - 1) / kBlockSize;

    if (tid == 0) {
        for (int i = 0; i < Sh::NSLOT; ++i) {
            mbar_init(full_bar(i), 1);
            mbar_init(empty_bar(i), 1);
        }
        mbar_init(s_bar(0), 1);
        mbar_init(s_bar(1), 1);
        mbar_init(p_bar, 128);
        mbar_init(o_bar, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) {
        tc::tmem_alloc(smem_addr(tmem_slot), Sh::TMEM_COLS);
        tc::tmem_relinquish();
    }

    // ---- Q tile -> shared memory, K-major with the 128-byte swizzle --------
    // row r = (token t0 + r / G, q head h*G + r % G); rows past the chunk and
    // the rows 128 - TPC*G that do not fill a token are zero
    {
        constexpr int CPR = D / 8;                // 16-byte chunks per row
        const T *qg = reinterpret_cast<const T *>(p.q);
        for (int idx = tid; idx < Sh::BM * CPR; idx += Sh::THREADS) {
            const int r = idx / CPR, ch = idx % CPR;
            const int tok = r / G, g = r % G;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < TPC * G && t0 + tok < c)
                v = __ldg(reinterpret_cast<const uint4 *>(
                    qg + ((size_t)(qs + t0 + tok) * Hq + h * G + g) * D + ch * 8));
            const int hf = ch >> 3, c8 = ch & 7;
            *reinterpret_cast<uint4 *>(smem + hf * (Sh::BM * 128) + r * 128 +
                                       ((c8 ^ (r & 7)) << 4)) = v;
        }
    }
    fence_proxy_async_shared();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    auto give_up = [&]() {
        *abort_flag = 1;
        record_error(p.err, PA_DEVERR_TIMEOUT);
    };

    if (warp == 0) {
        // ---------------- producer: K_j, V_j into the slot ring ----------------
        if (lane == 0) {
            const int32_t *table = p.block_tables + (size_t)s * p.max_blocks;
            int last[Sh::NSLOT] = {-1, -1, -1};
            for (int i = 0; i < 2 * nt; ++i) {
                if (*abort_flag)
                    break;
                const int j = i >> 1, sl = i % Sh::NSLOT;
                if (i >= Sh::NSLOT && !mbar_wait_bounded(empty_bar(sl), ((i / Sh::NSLOT) - 1) & 1)) {
                    give_up();
                    break;
                }
                int rows[4];
                int nv = 0;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int lb = 4 * j + b;
                    rows[b] = -1;
                    if (lb < nblk) {        // blocks past the sequence are not loaded
                        int phys = __ldg(table + lb);
                        if ((unsigned)phys >= (unsigned)p.num_blocks) {
                            record_error(p.err, PA_DEVERR_TABLE_RANGE);
                            phys = 0;
                        }
                        rows[b] = (phys * Hkv + h) * kBlockSize;
                        ++nv;
                    }
                }
                mbar_arrive_expect_tx(full_bar(sl), (uint32_t)(nv * Sh::HALVES * Sh::BOX));
                const void *tm = (i & 1) ? static_cast<const void *>(&tmv)
                                         : static_cast<const void *>(&tmk);
                const uint32_t dst = slot_addr + sl * Sh::SLOT_BYTES;
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    if (rows[b] >= 0)
#pragma unroll
                        for (int hf = 0; hf < Sh::HALVES; ++hf)
                            tma_load_2d(dst + (hf * 4 + b) * Sh::BOX, tm, 64 * hf, rows[b],
                                        full_bar(sl));
                last[sl] = i;
            }
            // every issued copy lands before the block may exit
            for (int sl = 0; sl < Sh::NSLOT; ++sl)
                if (last[sl] >= 0 &&
                    !mbar_wait_bounded(full_bar(sl), (last[sl] / Sh::NSLOT) & 1))
                    give_up();
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_f16(kBf16, Sh::BM, Sh::BN, false, false);
            constexpr uint32_t idO = tc::idesc_f16(kBf16, Sh::BM, D, false, true);
            auto issue_s = [&](int j) -> bool {
                const int i = 2 * j, sl = i % Sh::NSLOT;
                if (!mbar_wait_bounded(full_bar(sl), (i / Sh::NSLOT) & 1))
                    return false;
                tc::fence_after_sync();
                const uint32_t kb = slot_addr + sl * Sh::SLOT_BYTES;
                const uint32_t d = tmem + Sh::COL_S + (uint32_t)(j & 1) * Sh::BN;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t hf = k >> 2, w = (k & 3) * 32;
                    const uint64_t a = tc::sdesc_sw128(q_addr + hf * (Sh::BM * 128) + w, 16, 1024);
                    const uint64_t b = tc::sdesc_sw128(kb + hf * (4 * Sh::BOX) + w, 16, 1024);
                    tc::mma_ss(d, a, b, idS, k > 0);
                }
                tc::commit(s_bar(j & 1));
                tc::commit(empty_bar(sl));
                return true;
            };
            bool ok = issue_s(0);
            for (int j = 0; ok && j < nt; ++j) {
                if (*abort_flag) {
                    ok = false;
                    break;
                }
                if (j + 1 < nt && !issue_s(j + 1)) {
                    ok = false;
                    break;
                }
                const int i = 2 * j + 1, sl = i % Sh::NSLOT;
                if (!mbar_wait_bounded(p_bar, j & 1) ||
                    !mbar_wait_bounded(full_bar(sl), (i / Sh::NSLOT) & 1)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t vb = slot_addr + sl * Sh::SLOT_BYTES;
#pragma unroll
                for (int kk = 0; kk < Sh::BN / 16; ++kk) {
                    // A = P (K-major, keys 16kk..), B = V block kk (MN-major:
                    // 64-channel groups 4 boxes apart, 8-key groups 1 KB apart)
                    const uint64_t a = tc::sdesc_sw128(p_addr + kk * 32, 16, 1024);
                    const uint64_t b = tc::sdesc_sw128(vb + kk * Sh::BOX, 4 * Sh::BOX, 1024);
                    tc::mma_ss(tmem + Sh::COL_O, a, b, idO, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc::commit(o_bar);
                tc::commit(empty_bar(sl));
            }
            if (!ok)
                give_up();
            // no MMA may still run when TMEM is freed
            tc::commit(drain_bar);
            if (!mbar_wait_bounded(drain_bar, 0))
                give_up();
        }
    } else {
        // ---------------- softmax: one thread per row ----------------
        const int q4 = warp & 3;                   // TMEM lane quarter of this warp
        const int r = q4 * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        const int tok = r / G, g = r % G;
        const bool row_valid = r < TPC * G && t0 + tok < c;
        const int pos = row_valid ? L - c + t0 + tok : L - 1;
        float m = 0.f, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            if (__any_sync(FULL, *abort_flag != 0)) {
                ok = false;
                break;
            }
            if (!__all_sync(FULL, mbar_wait_bounded(s_bar(j & 1), (j >> 1) & 1))) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            __syncwarp();                        // tcgen05.ld is warp-collective
            float x[Sh::BN];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t v[32];
                tc::tmem_ld32(tmem + lane_off + Sh::COL_S + (uint32_t)(j & 1) * Sh::BN + 32 * half, v);
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    x[32 * half + e] = __uint_as_float(v[e]) * p.scale_log2;
            }
            const int k0 = j * Sh::BN;
            if (k0 + Sh::BN - 1 > pos) {
#pragma unroll
                for (int e = 0; e < Sh::BN; ++e)
                    if (k0 + e > pos)
                        x[e] = -INFINITY;   // causal mask (and keys >= L)
            }
            float mt = x[0];
#pragma unroll
            for (int e = 1; e < Sh::BN; ++e)
                mt = fmaxf(mt, x[e]);
            // O and P may be touched only after the previous P.V has completed
            if (j > 0) {
                if (!__all_sync(FULL, mbar_wait_bounded(o_bar, (j - 1) & 1))) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
            }
            bool grow = false;
            if (j == 0)
                m = mt;                  // finite: key 0 is visible to every row
            else
                grow = mt > m + 8.f;
            __syncwarp();
            if (__any_sync(FULL, grow)) {
                const float mn = grow ? mt : m;
                const float alpha = exp2f(m - mn);
                m = mn;
                l *= alpha;
#pragma unroll
                for (int cc = 0; cc < D; cc += 32) {
                    uint32_t v[32];
                    tc::tmem_ld32(tmem + lane_off + Sh::COL_O + cc, v);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                    tc::tmem_st32(tmem + lane_off + Sh::COL_O + cc, v);
                }
            }
            // the tile that reaches the end of the sequence: value rows of
            // keys >= L are zeroed (0 * NaN is NaN in the MMA)
            if (k0 + Sh::BN > L) {
                const int i = 2 * j + 1, sl = i % Sh::NSLOT;
                if (!__all_sync(FULL, mbar_wait_bounded(full_bar(sl), (i / Sh::NSLOT) & 1))) {
                    ok = false;
                    break;
                }
                // 128 threads of 4 warps zero the rows; their own barrier below
                // (p_bar) orders the stores before the MMA
                const int first = L - k0;
                const int n16 = (Sh::BN - first) * Sh::HALVES * 8;
                unsigned char *vb = smem + Sh::OFF_SLOT + sl * Sh::SLOT_BYTES;
                for (int idx = r; idx < n16; idx += 128) {
                    const int row = first + idx / (Sh::HALVES * 8);
                    const int rem = idx % (Sh::HALVES * 8);
                    *reinterpret_cast<uint4 *>(vb + ((rem >> 3) * 4 + (row >> 4)) * Sh::BOX +
                                               (row & 15) * 128 + (rem & 7) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
            }
            // P = exp2(x - m) as the A operand: row r, 8-key chunks swizzled
            float rs = 0.f;
            unsigned char *prow = smem + Sh::OFF_P + r * 128;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p0 = exp2f(x[8 * c8 + 2 * e] - m);
                    const float p1 = exp2f(x[8 * c8 + 2 * e + 1] - m);
                    rs += p0 + p1;
                    w[e] = Mma<T>::pack(p0, p1);
                }
                *reinterpret_cast<uint4 *>(prow + ((c8 ^ (r & 7)) << 4)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
            l += rs;
            fence_proxy_async_shared();
            tc::fence_before_sync();
            mbar_arrive(p_bar);
        }
        if (ok && !__all_sync(FULL, mbar_wait_bounded(o_bar, (nt - 1) & 1)))
            ok = false;
        if (ok) {
            tc::fence_after_sync();
            __syncwarp();
            const float inv = 1.f / l;
            T *orow = reinterpret_cast<T *>(p.out) +
                      ((size_t)(qs + t0 + tok) * Hq + h * G + g) * D;
#pragma unroll
            for (int cc = 0; cc < D; cc += 32) {
                uint32_t v[32];
                tc::tmem_ld32(tmem + lane_off + Sh::COL_O + cc, v);
                if (row_valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 u;
                        u.x = Mma<T>::pack(__uint_as_float(v[e]) * inv, __uint_as_float(v[e + 1]) * inv);
                        u.y = Mma<T>::pack(__uint_as_float(v[e + 2]) * inv, __uint_as_float(v[e + 3]) * inv);
                        u.z = Mma<T>::pack(__uint_as_float(v[e + 4]) * inv, __uint_as_float(v[e + 5]) * inv);
                        u.w = Mma<T>::pack(__uint_as_float(v[e + 6]) * inv, __uint_as_float(v[e + 7]) * inv);
                        *reinterpret_cast<uint4 *>(orow + cc + e) = u;
                    }
                }
            }
        } else {
            give_up();
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, Sh::TMEM_COLS);
    }
}

}  // namespace pa
