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
// One thread block (one per SM) computes 256 rows = (token, q head) pairs of
// one sequence and one kv head, as two 128-row query tiles ("groups") of
// 128 / G consecutive chunk tokens times the G q heads that share the kv
// head.  Both groups consume every K/V tile the block stages.
//
// Operand bytes per flop are kept low: key tiles of 128 (Q is read from
// shared memory once per 128 keys), and P never goes through shared memory
// -- the softmax writes it into tensor memory (over the score columns it has
// consumed, or at head_dim 64 into columns of its own), and P.V takes its A
// operand from there.  What bounds the kernel is each group's chain
// S -> softmax -> P.V -> next S against the other group's MMA work.
// Warp roles (320 threads):
//   warp 0    TMA producer of K and V tiles of 128 keys (8 pool blocks x 16
//             rows x 128-byte boxes) into a ring of slots;
//   warp 1    TMEM owner; issues the MMAs of both groups (the warp runs the
//             loop, one elected lane issues):
//               S_g,j = Q_g . K_j^T        (M 128, N 128, K = head_dim)
//               O_g  += P_g,j . V_j        (M 128, N head_dim, K 128; A in TMEM)
//             at head_dim 128 S_g,j+1 overwrites the columns P_g,j is read
//             from, so it is issued once P_g,j . V_j has completed; the two
//             groups alternate on the tensor core (one group's softmax runs
//             while the other group's MMAs do);
//   warps 2-5 group 0, warps 6-9 group 1: first load the Q tiles into
//             shared memory (while the producer's first K/V copies are in
//             flight); then one thread per row (its TMEM lane): scores from
//             TMEM, causal mask, online softmax in base 2 with a lazy
//             rescale of O (only when the running maximum grows by more than
//             2^8), P into TMEM, and the final O / l written out.
// TMEM (512 columns): group g uses [256g, 256g + 128) for S and
// [256g + 128, 256g + 128 + head_dim) for O.  P, packed two per column,
// overwrites S's first 64 columns at head_dim 128; at head_dim 64 it has the
// group's last 64 columns, and S_g,j+1 is then issued as soon as the softmax
// has read S_g,j.
// Every wait is bounded; a wait that gives up records PA_DEVERR_TIMEOUT and
// the block drains its copies and MMAs before it frees TMEM and exits.
#pragma once

#include <cuda.h>
#include <type_traits>

#include "pa_device.cuh"
#include "pa_prefill_abi.h"
#include "pa_tcgen05.cuh"

namespace pa {

template <int D>
struct PrefillShape {
    static constexpr int BM = kPrefillRows;                 // rows per group (tile)
    static constexpr int NG = kPrefillTiles;                // groups per block
    static constexpr int BN = kPrefillKeys;                 // keys per tile
    static constexpr int NB = BN / kBlockSize;              // pool blocks per tile
    static constexpr int HALVES = D / 64;                   // 128-byte column boxes
    static constexpr int BOX = 2048;                        // 16 rows x 128 B
    static constexpr int Q_BYTES = BM * D * 2;              // per group: [half][128 rows][128 B]
    static constexpr int SLOT_BYTES = BN * D * 2;           // [half][8 blocks][16 rows][128 B]
    static constexpr int NSLOT = (227 * 1024 - 1024 - NG * Q_BYTES) / SLOT_BYTES;   // K/V ring
    static constexpr int OFF_SLOT = NG * Q_BYTES;
    static constexpr int DATA = OFF_SLOT + NSLOT * SLOT_BYTES;   // 1024-aligned operand region
    // full[NSLOT] empty[NSLOT] s[2] p[2] o[2] drain q[2] read[2], then TMEM
    // base and abort flag
    static constexpr int NBAR = 2 * NSLOT + 5 * NG + 1;
    static constexpr int BAR_BYTES = NBAR * 8 + 8;
    // The operand region is aligned up to 1024 bytes inside the dynamic
    // allocation; the barriers sit in whichever end of the 1024-byte slack
    // has room.
    static constexpr int SMEM = DATA + 1024;
    static constexpr int THREADS = 64 + NG * 128;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t GROUP_COLS = 256;
    static constexpr uint32_t COL_S = 0;                    // S
    static constexpr uint32_t COL_O = 128;
    // P (BN/2 packed columns) gets its own columns when they fit beside S and
    // O (head_dim 64); otherwise it overwrites S's first half
    static constexpr bool SEPARATE_P = COL_O + D + BN / 2 <= GROUP_COLS;
    static constexpr uint32_t COL_P = SEPARATE_P ? COL_O + D : COL_S;
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(NSLOT >= 4, "at least two tiles of K/V in flight");
    static_assert(OFF_SLOT % 1024 == 0 && SLOT_BYTES % 1024 == 0, "swizzle atoms");
    static_assert(BAR_BYTES <= 512, "barriers fit either end of the slack");
    static_assert(SMEM <= 227 * 1024, "one block per SM");
};

// The (sequence, query tile, kv head) of block b under the work order;
// false past the end of the order.
__device__ __forceinline__ bool plan_block(const PrefillParams &p, int b, int &s, int &tile,
                                           int &h)
{
    const int Hkv = p.num_kv_heads;
    const int k = b / Hkv;
    if (k >= *p.plan_count)
        return false;
    uint32_t e = p.plan[k];
    if (*p.plan_by_seq) {
        const int s0 = (int)(e >> 16);
        const int st = p.plan_seq_start[s0], nq = p.plan_seq_nq[s0];
        const int local = b - Hkv * st;
        h = local / nq;
        e = p.plan[st + local % nq];
    } else {
        h = b % Hkv;
    }
    s = (int)(e >> 16);
    tile = (int)(e & 0xffffu);
    return true;
}

template <typename T, int D>
__global__ void __launch_bounds__(PrefillShape<D>::THREADS)
prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv)
{
    using Sh = PrefillShape<D>;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t FULL = 0xffffffffu;
    constexpr int NS = Sh::NSLOT;

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t slot_addr = sbase + Sh::OFF_SLOT;
    unsigned char *bars = (smem - smem_raw) >= Sh::BAR_BYTES ? smem_raw : smem + Sh::DATA;
    const uint32_t bar_addr = smem_addr(bars);
    auto full_bar = [&](int s) { return bar_addr + 8u * s; };
    auto empty_bar = [&](int s) { return bar_addr + 8u * (NS + s); };
    auto s_bar = [&](int g) { return bar_addr + 8u * (2 * NS + g); };
    auto p_bar = [&](int g) { return bar_addr + 8u * (2 * NS + Sh::NG + g); };
    auto o_bar = [&](int g) { return bar_addr + 8u * (2 * NS + 2 * Sh::NG + g); };
    const uint32_t drain_bar = bar_addr + 8u * (2 * NS + 3 * Sh::NG);
    auto q_bar = [&](int g) { return drain_bar + 8u * (1 + g); };   // Q_g is in shared memory
    // with P in its own columns: the group's softmax has read S_g,j
    auto read_bar = [&](int g) { return drain_bar + 8u * (1 + Sh::NG + g); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Sh::NBAR * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Hkv = p.num_kv_heads, Hq = p.num_heads, G = Hq / Hkv;
    const int TPG = Sh::BM / G;                   // chunk tokens per group
    const int TPB = Sh::NG * TPG;                 // chunk tokens per block
    int h = blockIdx.x % Hkv;

    // ---- the block's rows and key range (uniform over the block) ----------
    // no global memory is read before the preceding kernel (the plan) is done
    grid_dependency_wait();
    int s, rank = 0, tile = 0;
    if (p.plan) {
        if (!plan_block(p, blockIdx.x, s, tile, h))
            return;
    } else {
        const int per_rank = p.num_seqs * Hkv;
        rank = blockIdx.x / per_rank;
        s = (blockIdx.x % per_rank) / Hkv;
    }
    const int L = __ldg(p.seq_lens + s);
    const int qs = __ldg(p.query_start + s);
    const int c = __ldg(p.query_start + s + 1) - qs;
    const bool reporter = !p.plan && rank == 0 && h == 0 && tid == 0;   // the plan reports itself
    if (L < 0 || L > p.max_blocks * kBlockSize) {
        if (reporter)
            record_error(p.err, PA_DEVERR_SEQLEN_RANGE);
        return;
    }
    if (c < 0 || c > L) {
        if (reporter)
            record_error(p.err, PA_DEVERR_QUERY_RANGE);
        return;
    }
    if (!p.plan) {
        const int nq = (c + TPB - 1) / TPB;
        if (nq > p.q_ranks && reporter)
            record_error(p.err, PA_DEVERR_QUERY_RANGE);   // max_query_len too small
        if (rank >= nq)
            return;
        tile = nq - 1 - rank;                     // rank 0 = the last (longest) tile
    }
    const int t0 = tile * TPB;
    const int t_end = min(t0 + TPB, c);
    const int p_last = L - c + t_end - 1;         // position of the block's last row
    const int nt = p_last / Sh::BN + 1;           // key tiles (both groups)
    const int nblk = (L + kBlockSize - 1) / kBlockSize;

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(full_bar(i), 1);
            mbar_init(empty_bar(i), 1);
        }
        for (int g = 0; g < Sh::NG; ++g) {
            mbar_init(s_bar(g), 1);
            mbar_init(p_bar(g), 128);
            mbar_init(o_bar(g), 1);
        }
        mbar_init(drain_bar, 1);
        for (int g = 0; g < Sh::NG; ++g) {
            mbar_init(q_bar(g), Sh::NG * 128);
            mbar_init(read_bar(g), 128);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) {
        tc::tmem_alloc(smem_addr(tmem_slot), Sh::TMEM_COLS);
        tc::tmem_relinquish();
    }

    // the barriers and the TMEM base are visible to every thread; the Q
    // tiles are loaded by the softmax warps while K/V stream in
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
        // The whole warp works: lane l holds the pool row of block NB*win + l
        // of a window of WT tiles (the next window's entries are already in
        // flight), lane 0 waits for the slot and arms its barrier, and lanes
        // (hf, b) issue the tile's boxes in parallel.
        constexpr int NB = Sh::NB, WT = 32 / NB;
        const int32_t *table = p.block_tables + (size_t)s * p.max_blocks;
        auto fetch = [&](int w0) {
            const int lb = NB * w0 + lane;
            return lb < nblk ? __ldg(table + lb) : 0;
        };
        auto to_row = [&](int w0, int phys) {
            if (NB * w0 + lane >= nblk)
                return -1;                  // blocks past the sequence are not loaded
            if ((unsigned)phys >= (unsigned)p.num_blocks) {
                record_error(p.err, PA_DEVERR_TABLE_RANGE);
                phys = 0;
            }
            return (phys * Hkv + h) * kBlockSize;
        };
        int win = 0;
        int cur = to_row(0, fetch(0));
        int nxt = fetch(WT);
        int last = -1;                          // lane sl < NS: last item put in slot sl
        for (int i = 0; i < 2 * nt; ++i) {
            const int j = i >> 1, sl = i % NS;
            if (j == win + WT) {
                win += WT;
                cur = to_row(win, nxt);
                nxt = fetch(win + WT);
            }
            bool ready = true;
            if (lane == 0)
                ready = !*abort_flag &&
                        (i < NS || mbar_wait_bounded(empty_bar(sl), ((i / NS) - 1) & 1));
            if (!__shfl_sync(FULL, ready, 0)) {
                if (lane == 0 && !*abort_flag)
                    give_up();
                break;
            }
            const int nv = min(NB, nblk - NB * j);
            if (lane == 0)
                mbar_arrive_expect_tx(full_bar(sl), (uint32_t)(nv * Sh::HALVES * Sh::BOX));
            const int b = lane % NB, hf = lane / NB;
            const int row = __shfl_sync(FULL, cur, NB * (j - win) + b);
            __syncwarp();
            if (hf < Sh::HALVES && row >= 0) {
                const void *tm = (i & 1) ? static_cast<const void *>(&tmv)
                                         : static_cast<const void *>(&tmk);
                tma_load_2d(slot_addr + sl * Sh::SLOT_BYTES + (hf * NB + b) * Sh::BOX, tm,
                            64 * hf, row, full_bar(sl));
            }
            if (lane == sl)
                last = i;
        }
        // every issued copy lands before the block may exit
        if (lane < NS && last >= 0 && !mbar_wait_bounded(full_bar(lane), (last / NS) & 1))
            give_up();
    } else if (warp == 1) {
        // ---------------- MMA issuer (the whole warp, one elected lane issues) ------
        // The warp stays converged and every operand is warp-uniform, so the
        // descriptors live in uniform registers and the MMAs issue back to
        // back (a single-lane loop issues them at a fraction of the rate).
        constexpr uint32_t idS = tc::idesc_f16(kBf16, Sh::BM, Sh::BN, false, false);
        constexpr uint32_t idO = tc::idesc_f16(kBf16, Sh::BM, D, false, true);
        // descriptors of slot 0 / group 0; offsets are added in 16-byte units
        const uint64_t q_desc = tc::sdesc_sw128(sbase, 16, 1024);
        const uint64_t k_desc = tc::sdesc_sw128(slot_addr, 16, 1024);
        const uint64_t v_desc = tc::sdesc_sw128(slot_addr, Sh::NB * Sh::BOX, 1024);
        auto wait_all = [&](uint32_t bar, uint32_t parity) {
            return __all_sync(FULL, mbar_wait_bounded(bar, parity));
        };
        // S_g,j = Q_g . K_j^T; the K slot is released after the last group
        auto issue_s = [&](int g, int j) -> bool {
            const int i = 2 * j, sl = i % NS;
            if (!wait_all(full_bar(sl), (i / NS) & 1))
                return false;
            tc::fence_after_sync();
            const uint64_t qd = q_desc + (uint64_t)((g * Sh::Q_BYTES) >> 4);
            const uint64_t kd = k_desc + (uint64_t)((sl * Sh::SLOT_BYTES) >> 4);
            const uint32_t d = tmem + g * Sh::GROUP_COLS + Sh::COL_S;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                // K step k: 32 bytes along the 128-byte row; the next 64
                // channels are 16 KB further (Q: 128 rows, K: 8 boxes)
                const uint64_t ko = (uint64_t)(((k & 3) * 32 + (k >> 2) * (Sh::BM * 128)) >> 4);
                tc::mma_ss_warp(d, qd + ko, kd + ko, idS, k > 0);
            }
            tc::commit_warp(s_bar(g));
            if (g == Sh::NG - 1)
                tc::commit_warp(empty_bar(sl));
            return true;
        };
        static_assert(Sh::BM * 128 == Sh::NB * Sh::BOX, "Q and K halves 16 KB apart");
        // O_g += P_g,j . V_j once the group's softmax has written P
        auto issue_pv = [&](int g, int j) -> bool {
            const int i = 2 * j + 1, sl = i % NS;
            if (!wait_all(p_bar(g), j & 1) || !wait_all(full_bar(sl), (i / NS) & 1))
                return false;
            tc::fence_after_sync();
            const uint64_t vd = v_desc + (uint64_t)((sl * Sh::SLOT_BYTES) >> 4);
            const uint32_t gc = tmem + g * Sh::GROUP_COLS;
#pragma unroll
            for (int kk = 0; kk < Sh::BN / 16; ++kk) {
                // A = P: keys 16kk.. = 8 packed columns; B = V block kk
                // (MN-major: 64-channel groups NB boxes apart, 8-key groups
                // 1 KB apart)
                tc::mma_ts_warp(gc + Sh::COL_O, gc + Sh::COL_P + 8 * kk,
                                vd + (uint64_t)((kk * Sh::BOX) >> 4), idO,
                                (j > 0 || kk > 0) ? 1u : 0u);
            }
            tc::commit_warp(o_bar(g));
            if (g == Sh::NG - 1)
                tc::commit_warp(empty_bar(sl));
            return true;
        };
        // while this block's query rows load: warm L2 with those of the
        // block one wave later (its pair and kv head from the work order)
        if (p.plan) {
            int s2, tile2, h2;
            if (plan_block(p, (int)blockIdx.x + p.wave, s2, tile2, h2)) {
                const int qs2 = __ldg(p.query_start + s2);
                const int t02 = tile2 * TPB;
                const int ntok = min(TPB, __ldg(p.query_start + s2 + 1) - qs2 - t02);
                const int lines = G * D * 2 / 128;  // 128-byte lines of a token's G heads
                const T *qg = reinterpret_cast<const T *>(p.q);
                for (int i = lane; i < ntok * lines; i += 32)
                    prefetch_l2(qg + ((size_t)(qs2 + t02 + i / lines) * Hq + h2 * G) * D +
                                (i % lines) * 64);
            }
        }
        bool ok = true;
        for (int g = 0; ok && g < Sh::NG; ++g)
            ok = wait_all(q_bar(g), 0) && issue_s(g, 0);
        for (int j = 0; ok && j < nt; ++j) {
            if (__any_sync(FULL, *abort_flag != 0)) {
                ok = false;
                break;
            }
            for (int g = 0; ok && g < Sh::NG; ++g) {
                if constexpr (Sh::SEPARATE_P) {
                    // S_g,j+1 only needs the softmax to have read S_g,j
                    if (j + 1 < nt)
                        ok = wait_all(read_bar(g), j & 1) && issue_s(g, j + 1);
                    ok = ok && issue_pv(g, j);
                } else {
                    ok = issue_pv(g, j);
                    // S_g,j+1 reuses the TMEM columns P_g,j . V_j reads
                    if (ok && j + 1 < nt)
                        ok = wait_all(o_bar(g), j & 1) && issue_s(g, j + 1);
                }
            }
        }
        if (!ok && lane == 0)
            give_up();
        // no MMA may still run when TMEM is freed
        tc::commit_warp(drain_bar);
        if (!wait_all(drain_bar, 0) && lane == 0)
            give_up();
    } else {
        // ---------------- Q tiles -> shared memory ----------------
        // K-major with the 128-byte swizzle.  Row rr of group g = (token
        // t0 + g*TPG + rr / G, q head h*G + rr % G); rows past the chunk and
        // the rows 128 - TPG*G that do not fill a token are zero.  Thread lt
        // takes 16-byte chunk lt % CPR of every (NG*128 / CPR)-th row, group
        // 0's rows first, with all its loads in flight at once; it arrives on
        // q_bar(g) once its rows of group g are stored, and the MMA warp
        // issues S_g,0 after that barrier.
        {
            constexpr int CPR = D / 8;            // 16-byte chunks per row
            constexpr int RSTEP = Sh::NG * 128 / CPR;
            constexpr int NPT = Sh::NG * Sh::BM / RSTEP;
            constexpr int PER_G = NPT / Sh::NG;   // a thread's chunks in each group
            const T *qg = reinterpret_cast<const T *>(p.q);
            const int lt = tid - 64, ch = lt % CPR, hf = ch >> 3, c8 = ch & 7;
            uint4 qv[NPT];
#pragma unroll
            for (int i = 0; i < NPT; ++i) {
                const int r = lt / CPR + i * RSTEP;
                const int g = r / Sh::BM, rr = r % Sh::BM;
                const int tok = g * TPG + rr / G, hg = rr % G;
                qv[i] = make_uint4(0, 0, 0, 0);
                if (rr < TPG * G && t0 + tok < c)
                    qv[i] = __ldg(reinterpret_cast<const uint4 *>(
                        qg + ((size_t)(qs + t0 + tok) * Hq + h * G + hg) * D + ch * 8));
            }
#pragma unroll
            for (int i = 0; i < NPT; ++i) {
                const int r = lt / CPR + i * RSTEP;
                const int g = r / Sh::BM, rr = r % Sh::BM;
                *reinterpret_cast<uint4 *>(smem + g * Sh::Q_BYTES + hf * (Sh::BM * 128) +
                                           rr * 128 + ((c8 ^ (rr & 7)) << 4)) = qv[i];
                if (i % PER_G == PER_G - 1) {
                    fence_proxy_async_shared();
                    mbar_arrive(q_bar(i / PER_G));
                }
            }
        }
        static_assert(Sh::THREADS == 64 + Sh::NG * 128 && (Sh::NG * 128) % (D / 8) == 0 &&
                          (Sh::NG * Sh::BM) % (Sh::NG * 128 / (D / 8)) == 0,
                      "Q chunks divide evenly over the softmax warps");
        static_assert((Sh::BM * (D / 8)) % (Sh::NG * 128) == 0 &&
                          Sh::BM % (Sh::NG * 128 / (D / 8)) == 0,
                      "each thread's chunks of a group are consecutive in its loop");

        // ---------------- softmax: one thread per row of its group ----------
        const int grp = (warp - 2) >> 2;
        const int q4 = warp & 3;                   // TMEM lane quarter of this warp
        const int rr = q4 * 32 + lane;             // row within the group
        const uint32_t tg = tmem + ((uint32_t)(q4 * 32) << 16) + grp * Sh::GROUP_COLS;
        const int tok = grp * TPG + rr / G, hg = rr % G;
        const bool row_valid = rr < TPG * G && t0 + tok < c;
        const int pos = row_valid ? L - c + t0 + tok : L - 1;
        const float sl2 = p.scale_log2;
        float m = 0.f, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            if (__any_sync(FULL, *abort_flag != 0)) {
                ok = false;
                break;
            }
            if (!__all_sync(FULL, mbar_wait_bounded(s_bar(grp), j & 1))) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            const int k0 = j * Sh::BN;
            const int vis = pos - k0;              // keys [0, vis] of the tile are visible
            // the 128 scores of the row, both halves held in registers
            uint32_t v[2][64];
            __syncwarp();                        // tcgen05.ld is warp-collective
            tc::tmem_ld64(tg + Sh::COL_S, v[0]);
            tc::tmem_ld64(tg + Sh::COL_S + 64, v[1]);
            if constexpr (Sh::SEPARATE_P) {
                tc::fence_before_sync();
                mbar_arrive(read_bar(grp));      // S_g,j+1 may go in
            }
            // tiles left of the diagonal (the common case) need no mask
            const bool full = __all_sync(FULL, vis >= Sh::BN - 1);
            if (!full) {
#pragma unroll
                for (int e = 0; e < Sh::BN; ++e)
                    if (e > vis)
                        v[e >> 6][e & 63] = __float_as_uint(-INFINITY);
            }
            // row maximum as a tree, three operands per instruction
            float mx[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                auto x = [&](int i) { return __uint_as_float(v[i >> 6][i & 63]); };
                float t = fmax3(x(a), x(a + 8), x(a + 16));
#pragma unroll
                for (int i = a + 24; i < 120; i += 16)
                    t = fmax3(t, x(i), x(i + 8));
                mx[a] = fmaxf(t, x(a + 120));
            }
            float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                             fmaxf(mx[6], mx[7]));
            mt *= sl2;                           // scale > 0: max commutes with it
            // running maximum, raised lazily: only when the tile's maximum
            // exceeds it by more than 8 (P stays below 2^8 otherwise)
            bool grow = false;
            float alpha = 1.f;
            if (j == 0) {
                m = mt;                          // finite: key 0 is visible to every row
            } else if (mt > m + 8.f) {
                grow = true;
                alpha = ex2_approx(m - mt);
                m = mt;
            }
            // P = 2^(scale*s - m) packed to the operand type, written into
            // TMEM over score columns already read: keys 0-63 -> columns
            // 0-31, keys 64-127 -> 32-63.  Scale-and-subtract and the row sum
            // run two values per instruction.
            if constexpr (Sh::SEPARATE_P) {
                // P_g,j overwrites P_g,j-1, and O may be rescaled below: both
                // wait for P_g,j-1 . V_j-1 (with P apart from S, S_g,j was
                // issued without it)
                if (j > 0 && !__all_sync(FULL, mbar_wait_bounded(o_bar(grp), (j - 1) & 1))) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
            }
            const uint64_t sl2x2 = f2_pack(sl2, sl2), nmx2 = f2_pack(-m, -m);
            uint64_t sum2[4] = {0, 0, 0, 0};
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                uint32_t pw[32];
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    float y0, y1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(v[hb][e]), __uint_as_float(v[hb][e + 1])),
                                     sl2x2, nmx2),
                              y0, y1);
                    const float p0 = ex2_approx(y0);
                    const float p1 = ex2_approx(y1);
                    sum2[(e >> 1) & 3] = f2_add(sum2[(e >> 1) & 3], f2_pack(p0, p1));
                    pw[e / 2] = Mma<T>::pack(p0, p1);
                }
                __syncwarp();
                tc::tmem_st32(tg + Sh::COL_P + 32 * hb, pw);
            }
            float sum[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float a, b;
                f2_unpack(sum2[q], a, b);
                sum[q] = a + b;
            }
            l = fmaf(l, alpha, (sum[0] + sum[1]) + (sum[2] + sum[3]));
            // the tile that reaches the end of the sequence: value rows of
            // keys >= L are zeroed (0 * NaN is NaN in the MMA).  Group 0 does
            // it; group 1's P.V is issued after group 0's barrier, which
            // orders these stores before it.
            if (grp == 0 && k0 + Sh::BN > L) {
                const int i = 2 * j + 1, sl = i % NS;
                if (!__all_sync(FULL, mbar_wait_bounded(full_bar(sl), (i / NS) & 1))) {
                    ok = false;
                    break;
                }
                const int first = L - k0;
                const int n16 = (Sh::BN - first) * Sh::HALVES * 8;
                unsigned char *vb = smem + Sh::OFF_SLOT + sl * Sh::SLOT_BYTES;
                for (int idx = rr; idx < n16; idx += 128) {
                    const int row = first + idx / (Sh::HALVES * 8);
                    const int rem = idx % (Sh::HALVES * 8);
                    *reinterpret_cast<uint4 *>(vb + ((rem >> 3) * Sh::NB + (row >> 4)) * Sh::BOX +
                                               (row & 15) * 128 + (rem & 7) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_shared();
            }
            // O rescale: P_g,j-1 . V_j-1 has completed (before S_g,j was
            // issued, or, with P in its own columns, by the wait above)
            __syncwarp();
            if (__any_sync(FULL, grow)) {
#pragma unroll
                for (int cc = 0; cc < D; cc += 32) {
                    uint32_t v[32];
                    tc::tmem_ld32(tg + Sh::COL_O + cc, v);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                    tc::tmem_st32(tg + Sh::COL_O + cc, v);
                }
            }
            tc::fence_before_sync();
            mbar_arrive(p_bar(grp));
        }
        if (ok && !__all_sync(FULL, mbar_wait_bounded(o_bar(grp), (nt - 1) & 1)))
            ok = false;
        if (ok) {
            tc::fence_after_sync();
            __syncwarp();
            const float inv = 1.f / l;
            T *orow = reinterpret_cast<T *>(p.out) +
                      ((size_t)(qs + t0 + tok) * Hq + h * G + hg) * D;
#pragma unroll
            for (int cc = 0; cc < D; cc += 32) {
                uint32_t v[32];
                tc::tmem_ld32(tg + Sh::COL_O + cc, v);
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

// ---------------------------------------------------------------------------
// Work order of a prefill, one block.  The hardware hands thread blocks to
// SMs in index order as SMs free up, so the order decides both the schedule
// and what the blocks running at the same time share (plan_block maps a
// block to its work):
//  * the (sequence, query tile) pairs sorted by their key-tile count,
//    heaviest first (a counting sort on the count), block b taking pair
//    plan[b / Hkv] for kv head b % Hkv: the greedy longest-first schedule,
//    ending on the lightest pairs.  Used when the batch's K/V fits in L2, so
//    any blocks may run side by side;
//  * otherwise sequence by sequence, the sequences ordered by their heaviest
//    tile and each sequence's tiles heaviest first; a sequence's blocks take
//    its kv heads one after the other, each with all of its query tiles.
//    The blocks running at one time then stream the K/V of a few kv heads of
//    one sequence, together, so L2 serves the re-reads and each head's K/V
//    leaves DRAM about once.
// Pairs of one count keep no particular order (their results do not depend
// on it).
// ---------------------------------------------------------------------------
constexpr int kPlanBuckets = 2048;   // key-tile counts above this share the top bucket

__global__ void __launch_bounds__(1024)
prefill_plan_kernel(const PrefillParams p, int tpb, int bn, uint32_t *plan, int *count,
                    long long kv_bytes_per_token, long long l2_bytes, int *by_seq,
                    int32_t *seq_start, int32_t *seq_nq)
{
    __shared__ int hist_tile[kPlanBuckets];  // pairs per key-tile count
    __shared__ int hist_seq[kPlanBuckets];   // pairs of the sequences whose heaviest tile has it
    __shared__ unsigned long long tokens;
    const int tid = threadIdx.x, lane = tid & 31;
    grid_dependents_launch();                // the prefill may be scheduled; it waits for us
    for (int i = tid; i < kPlanBuckets; i += 1024) {
        hist_tile[i] = 0;
        hist_seq[i] = 0;
    }
    if (tid == 0)
        tokens = 0;
    __syncthreads();
    // the query tiles of sequence s that run: [first, last); errors reported once
    auto tiles = [&](int s, bool report, int &L, int &c, int &first) {
        L = p.seq_lens[s];
        const int qs = p.query_start[s];
        c = p.query_start[s + 1] - qs;
        first = 0;
        if (L < 0 || L > p.max_blocks * kBlockSize) {
            if (report)
                record_error(p.err, PA_DEVERR_SEQLEN_RANGE);
            return 0;
        }
        if (c < 0 || c > L) {
            if (report)
                record_error(p.err, PA_DEVERR_QUERY_RANGE);
            return 0;
        }
        const int nq = (c + tpb - 1) / tpb;
        if (nq > p.q_ranks) {                // the grid covers the last q_ranks tiles
            if (report)
                record_error(p.err, PA_DEVERR_QUERY_RANGE);
            first = nq - p.q_ranks;
        }
        return nq;
    };
    auto bucket = [&](int L, int c, int t) {
        const int t_end = min((t + 1) * tpb, c);
        return min((L - c + t_end - 1) / bn + 1, kPlanBuckets - 1);
    };
    // pass 1: both histograms and the batch's token count; a thread keeps
    // its first sequence's tiles in registers for pass 2 (every sequence
    // when num_seqs <= 1024)
    int L0 = 0, c0 = 0, first0 = 0, nq0 = 0;
    unsigned long long my_tokens = 0;
    for (int s = tid; s < p.num_seqs; s += 1024) {
        int L, c, first;
        const int nq = tiles(s, true, L, c, first);
        if (s == tid) {
            L0 = L;
            c0 = c;
            first0 = first;
            nq0 = nq;
        }
        for (int t = first; t < nq; ++t)
            atomicAdd(&hist_tile[bucket(L, c, t)], 1);
        if (nq > first) {
            atomicAdd(&hist_seq[bucket(L, c, nq - 1)], nq - first);
            my_tokens += (unsigned long long)L;
        }
    }
    if (my_tokens)
        atomicAdd(&tokens, my_tokens);
    __syncthreads();
    const bool by_sequence = (long long)tokens * kv_bytes_per_token > l2_bytes;
    if (tid == 0)
        *by_seq = by_sequence ? 1 : 0;
    int *hist = by_sequence ? hist_seq : hist_tile;
    // start of each bucket in descending order of the count: thread t owns
    // buckets B-1-2t and B-2-2t; warp scans, then a scan of the warp totals
    {
        __shared__ int warp_sum[32];
        static_assert(kPlanBuckets == 2 * 1024, "two buckets per thread");
        const int hi = kPlanBuckets - 1 - 2 * tid;
        const int n0 = hist[hi], n1 = hist[hi - 1];
        int incl = n0 + n1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += y;
        }
        if (lane == 31)
            warp_sum[tid >> 5] = incl;
        __syncthreads();
        if (tid < 32) {
            const int own = warp_sum[lane];
            int w = own;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o)
                    w += y;
            }
            warp_sum[lane] = w - own;            // exclusive
            if (lane == 31)
                *count = w;
        }
        __syncthreads();
        const int start = warp_sum[tid >> 5] + incl - (n0 + n1);
        hist[hi] = start;
        hist[hi - 1] = start + n0;
    }
    __syncthreads();
    for (int s = tid; s < p.num_seqs; s += 1024) {
        int L = L0, c = c0, first = first0, nq = nq0;
        if (s != tid)
            nq = tiles(s, false, L, c, first);
        if (by_sequence) {
            if (nq > first) {
                int at = atomicAdd(&hist_seq[bucket(L, c, nq - 1)], nq - first);
                seq_start[s] = at;
                seq_nq[s] = nq - first;
                for (int t = nq - 1; t >= first; --t)
                    plan[at++] = ((uint32_t)s << 16) | (uint32_t)t;
            }
        } else {
            for (int t = first; t < nq; ++t)
                plan[atomicAdd(&hist_tile[bucket(L, c, t)], 1)] = ((uint32_t)s << 16) | (uint32_t)t;
        }
    }
}

}  // namespace pa
