// pa_schedule.cuh -- how a decode's work is cut and handed to thread blocks.
//
// The work is a flat list of (sequence, kv head, 16-token tile) units ordered
// by sequence, then kv head, then tile.  A persistent grid walks it:
//  * balanced mode: thread block b owns the tile range [b*R, (b+1)*R), R the
//    tiles divided evenly over the grid, so every block reads the same bytes
//    whatever the length mix; a (sequence, kv head) run cut by a range
//    boundary leaves partial results that the log-sum-exp merge combines
//    (split-K along the sequence, FlashDecoding in the ICML tutorial notes,
//    section "内核优化");
//  * fixed mode: the units are partitions of part_tiles tiles of one run,
//    handed out in balanced contiguous ranges of partitions;
//  * whole mode: the units are whole runs (no split).
// Every thread of a block evaluates the walker identically, so the pieces it
// yields are block-uniform.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

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

}  // namespace pa
