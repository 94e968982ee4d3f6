// pa_schedule.cuh -- how a decode's work is cut and handed to warps.
//
// The work is a flat list of (sequence, kv head, 16-token tile) units ordered
// by sequence, then kv head, then tile; the tiles of one (sequence, kv head)
// form a "run".  Every warp of the persistent grid is an independent worker
// that walks its own part of the list, so warps never wait for each other:
//  * balanced mode: worker k owns the tile range [k*R, (k+1)*R), R the tiles
//    divided evenly over all workers, so every worker reads the same bytes
//    whatever the length mix.  A run cut by a range boundary leaves partial
//    results that a log-sum-exp merge combines (split-K along the sequence,
//    FlashDecoding in the ICML tutorial notes, section "内核优化").
//  * fixed mode: the same ranges, with runs also cut at partition boundaries
//    (part_tiles tiles); each partition's partial result is the split-K unit,
//    merged per run afterwards.
//  * whole mode: worker k owns whole runs (no split), an even share by count.
// A "piece" is the part of one run (and, in fixed mode, of one partition) that
// lies in one worker's range: tiles [tb, te) of run (s, h).
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

struct Walker {
    // constants
    const int32_t *pre;   // prefix over sequences of tiles (whole mode: of non-empty runs' sequences)
    const int32_t *lens;  // clamped lengths [n]
    int n, hkv, mode, pt;
    int R;                // tiles per worker (balanced / fixed)
    // state
    int s, h, tb, te, nt;
    int F;                // flat index of tile 0 of run (s, h)
    int A, B;             // this worker's flat tile range, or run-index range (whole mode)
    int cur;              // whole mode: current run index
    int part;             // fixed mode: partition of the current piece
    bool valid;
    bool first;           // first piece of this worker

    __device__ __forceinline__ int tiles_of(int seq) const
    {
        return (lens[seq] + kBlockSize - 1) / kBlockSize;
    }

    // largest s with hkv * pre[s] <= x (sequences without units are skipped)
    __device__ __forceinline__ int find_seq(int x) const
    {
        int lo = 0, hi = n - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (hkv * pre[mid] <= x)
                lo = mid;
            else
                hi = mid - 1;
        }
        return lo;
    }

    // piece end inside run (s, h) starting at tile tb
    __device__ __forceinline__ void close_piece()
    {
        te = min(nt, B - F);
        if (mode == kModeFixed) {
            part = tb / pt;
            te = min(te, (part + 1) * pt);
        }
    }

    __device__ __forceinline__ void init(const int32_t *pre_, const int32_t *lens_, int n_,
                                         int hkv_, int mode_, int pt_, int min_tiles, int workers,
                                         int k)
    {
        pre = pre_;
        lens = lens_;
        n = n_;
        hkv = hkv_;
        mode = mode_;
        pt = pt_;
        first = true;
        part = 0;
        const int total = hkv * pre[n];          // tiles, or non-empty runs in whole mode
        if (mode == kModeWhole) {
            A = (int)((long long)k * total / workers);
            B = (int)((long long)(k + 1) * total / workers);
            valid = A < B;
            if (!valid)
                return;
            cur = A;
            s = find_seq(A);
            h = A - hkv * pre[s];
            nt = tiles_of(s);
            F = 0;
            tb = 0;
            te = nt;
            return;
        }
        R = max((total + workers - 1) / workers, min_tiles);
        const long long a = (long long)k * R;
        valid = a < total;
        if (!valid)
            return;
        A = (int)a;
        B = min(total, A + R);
        s = find_seq(A);
        nt = pre[s + 1] - pre[s];
        h = (A - hkv * pre[s]) / nt;
        F = hkv * pre[s] + h * nt;
        tb = A - F;
        close_piece();
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
        if (mode == kModeWhole) {
            if (++cur >= B) {
                valid = false;
                return;
            }
            if (++h == hkv) {
                h = 0;
                next_seq();
                nt = tiles_of(s);
            }
            tb = 0;
            te = nt;
            return;
        }
        if (F + te >= B) {
            valid = false;
            return;
        }
        if (te < nt) {           // fixed mode: next partition of the same run
            tb = te;
        } else {                 // next run
            F += nt;
            if (++h == hkv) {
                h = 0;
                next_seq();
                nt = pre[s + 1] - pre[s];
            }
            tb = 0;
        }
        close_piece();
    }

    // the piece is the whole run
    __device__ __forceinline__ bool whole_run() const { return tb == 0 && te == nt; }

    // fixed mode: the piece is a whole partition
    __device__ __forceinline__ bool whole_part() const
    {
        return mode == kModeFixed && tb == part * pt && te == min(nt, (part + 1) * pt);
    }
};

// Units a sequence of (clamped) length L contributes to the flat list.
__device__ __forceinline__ int seq_units(int L, int mode)
{
    const int nt = (L + kBlockSize - 1) / kBlockSize;
    return mode == kModeWhole ? (nt > 0 ? 1 : 0) : nt;
}

// Clamp the lengths and build the exclusive unit prefix (into shared memory
// in the decode kernel, into the workspace in the prep kernel for large
// batches).  Also flag each sequence whose first block is named by a
// neighbouring sequence's table too (share[s] = 1): sequences forked from one
// prompt (parallel samples) share their prompt's blocks and sit next to each
// other in the batch.  Only flagged sequences pay for per-tile sharing checks.
// This builds sequences [begin, end) with the prefix counted from begin
// (neighbours are looked up in the whole batch), leaves the range's unit
// count in *total and returns whether any of this thread's sequences is
// flagged; pre[end] is not written.
//
// The block walks the range in rows of K * NT consecutive sequences, thread
// t taking sequences row + K t .. row + K t + K - 1, so a warp's loads cover
// one contiguous stretch (a thread owning a long run of consecutive
// sequences made each warp load touch 32 cache lines).  The neighbours at a
// thread's ends come from the adjacent lanes by shuffle, at a warp's ends
// from plain loads.  Each row's units are scanned across the block and added
// to the running total of the rows before it; RW rows' loads are issued at
// once.  The large-batch prep kernels take K = 4 (one row of 1024
// sequences a block); a decode block, whose batch is at most a few rows,
// K = 1 (with K = 4 one warp would hold a small batch's every sequence).
template <int NT, int K, int RW>
__device__ __forceinline__ bool build_prefix(const DecodeParams &p, int begin, int end,
                                             int32_t *pre, int32_t *lens, uint8_t *share,
                                             int *total_out)
{
    constexpr int NW = NT / 32;
    constexpr int ROW = K * NT;
    constexpr uint32_t FULL = 0xffffffffu;
    __shared__ int warp_sum[NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = p.num_seqs;
    const int maxlen = p.max_blocks * kBlockSize;
    const size_t mb = (size_t)p.max_blocks;
    int carry = 0;
    bool bad = false, any = false;
    for (int base = begin; base < end; base += RW * ROW) {
        // every load below is in bounds whatever the lengths hold
        int Lr[RW][K], br[RW][K], Le[RW], be[RW];
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            const int s0 = base + r * ROW + K * tid;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int s = s0 + k;
                Lr[r][k] = 0;
                br[r][k] = -1;
                if (s < n) {
                    Lr[r][k] = __ldg(p.seq_lens + s);
                    br[r][k] = __ldg(p.block_tables + s * mb);
                }
            }
            // the warp's ends: lane 0 needs sequence s0 - 1, lane 31 s0 + K
            const int e = lane == 0 ? s0 - 1 : s0 + K;
            Le[r] = 0;
            be[r] = -1;
            if ((lane == 0 || lane == 31) && e >= 0 && e < n) {
                Le[r] = __ldg(p.seq_lens + e);
                be[r] = __ldg(p.block_tables + e * mb);
            }
        }
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            const int row = base + r * ROW;
            if (row >= end)
                break;                                   // the same for the whole block
            const int s0 = row + K * tid;
            // raw neighbour values (a sequence past the end reads as empty)
            int Lp = __shfl_up_sync(FULL, Lr[r][K - 1], 1);
            int bp = __shfl_up_sync(FULL, br[r][K - 1], 1);
            int Ln = __shfl_down_sync(FULL, Lr[r][0], 1);
            int bn = __shfl_down_sync(FULL, br[r][0], 1);
            if (lane == 0) {
                Lp = Le[r];
                bp = be[r];
            }
            if (lane == 31) {
                Ln = Le[r];
                bn = be[r];
            }
            int u[K], sum = 0;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int s = s0 + k;
                u[k] = 0;
                if (s < end) {
                    int L = Lr[r][k];
                    if (L < 0 || L > maxlen) {
                        bad = true;
                        L = L < 0 ? 0 : maxlen;
                    }
                    const int lp = k > 0 ? Lr[r][k - 1] : Lp, bpk = k > 0 ? br[r][k - 1] : bp;
                    const int ln = k + 1 < K ? Lr[r][k + 1] : Ln;
                    const int bnk = k + 1 < K ? br[r][k + 1] : bn;
                    const bool sh = L > 0 && ((lp > 0 && bpk == br[r][k]) ||
                                              (ln > 0 && bnk == br[r][k]));
                    lens[s] = L;
                    share[s] = (uint8_t)sh;
                    any |= sh;
                    u[k] = seq_units(L, p.mode);
                }
                sum += u[k];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(FULL, incl, o);
                if (lane >= o)
                    incl += y;
            }
            if (lane == 31)
                warp_sum[warp] = incl;
            __syncthreads();
            int before = 0, total = 0;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const int x = warp_sum[w];
                before += w < warp ? x : 0;
                total += x;
            }
            int run = carry + before + incl - sum;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                if (s0 + k < end)
                    pre[s0 + k] = run;
                run += u[k];
            }
            carry += total;
            __syncthreads();                             // warp_sum is reused
        }
    }
    if (bad && (blockIdx.x == 0 || begin > 0))
        record_error(p.err, PA_DEVERR_SEQLEN_RANGE);
    *total_out = carry;
    return any;
}

// A cut unit (a run in balanced mode, a partition in fixed mode) as recorded
// by the worker in whose range it starts, for the merge.
struct CutDesc {
    int s, h, part, u0;   // sequence, kv head, partition, flat index of the unit's first tile
    int nu, R, np, valid; // tiles of the unit, tiles per worker, partitions of the run, flag
};

// The pieces of a cut unit [u0, u0 + nu) whose descriptor is worker c0's:
// one in each of workers c0 .. cut_last_worker; worker c's piece is in its
// first slot (2c), except worker c0's when the unit starts inside its range
// (c0_last: its last slot, 2c0 + 1).
__device__ __forceinline__ int cut_last_worker(int u0, int nu, int R)
{
    return (u0 + nu - 1) / R;
}

__device__ __forceinline__ int cut_piece_slot(int c, int c0, bool c0_last)
{
    return (c == c0 && c0_last) ? 2 * c + 1 : 2 * c;
}

}  // namespace pa
