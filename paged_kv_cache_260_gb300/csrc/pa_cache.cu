// pa_cache.cu -- kernels that maintain the KV block pool, plus the debug
// gather and the table check.  All of them are raw 16-byte copies: the
// element type does not matter, only head_dim * 2 bytes per row.
#include "pa_cache.h"
#include "pa_device.cuh"

namespace pa {

// ---------------------------------------------------------------------------
// reshape_and_cache: token i's K/V rows (all kv heads) -> pool slot
// slot_mapping[i].  The input is read as one flat run of 16-byte vectors (K of
// every token, then V); a row of head_dim * 2 bytes is 2^row_shift vectors.
// A block takes U * blockDim.x consecutive vectors at a time, each thread U of
// them blockDim.x apart: every load instruction of a warp is coalesced, and a
// thread has its U loads in flight before its stores.  (Striding a thread's
// vectors across the whole grid instead spreads a warp over U distant regions
// and ran 11 % slower on a bulk write.)
// ---------------------------------------------------------------------------
template <int U>
__global__ void __launch_bounds__(256)
reshape_and_cache_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                         uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                         const int64_t *__restrict__ slot_mapping, int num_tokens,
                         int num_kv_heads, int row_shift, long long num_slots, uint32_t *err)
{
    grid_dependents_launch();   // a dependent decode may be scheduled now; it waits for us
    using idx = unsigned long long;                 // unsigned: the divisions stay cheap
    const idx half = ((idx)num_tokens * (idx)num_kv_heads) << row_shift;  // vectors of K
    const idx total = 2 * half;
    const idx vmask = ((idx)1 << row_shift) - 1;
    const idx heads = (idx)num_kv_heads;
    const idx step = (idx)gridDim.x * blockDim.x * U;
    for (idx base = (idx)blockIdx.x * blockDim.x * U + threadIdx.x; base < total; base += step) {
        uint4 t[U];
        uint4 *to[U];                                     // null: nothing to store
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const idx x = base + (idx)u * blockDim.x;
            to[u] = nullptr;
            if (x >= total)
                continue;
            const bool is_v = x >= half;
            const idx y = is_v ? x - half : x;            // vector within K (or V)
            const idx row = y >> row_shift;
            const idx i = row / heads;                    // token
            const idx kvh = row - i * heads;
            const int64_t slot = __ldg(slot_mapping + i);
            t[u] = __ldg((is_v ? v_new : k_new) + y);
            if (slot < 0)
                continue;                                 // padding token
            if (slot >= num_slots) {
                if ((y & vmask) == 0 && kvh == 0 && !is_v)
                    record_error(err, PA_DEVERR_SLOT_RANGE);
                continue;
            }
            const idx blk = (idx)slot / kBlockSize, off = (idx)slot % kBlockSize;
            const idx dst = (((blk * heads + kvh) * kBlockSize + off) << row_shift) + (y & vmask);
            to[u] = (is_v ? v_cache : k_cache) + dst;
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (to[u])
                *to[u] = t[u];
    }
}

// ---------------------------------------------------------------------------
// Whole-block copies between pools: copy_blocks (copy-on-write, within one
// pool) and swap_blocks (between the GPU pool and a pool in pinned host
// memory, reached over the C2C link).  blockIdx.y picks the pair and K or V;
// each thread moves 4 vectors 256 apart (4 loads in flight).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
copy_blocks_kernel(uint4 *dst_k, uint4 *dst_v, const uint4 *src_k, const uint4 *src_v,
                   const int64_t *__restrict__ block_mapping, int num_pairs, long long block_vecs,
                   long long src_blocks, long long dst_blocks, uint32_t *err)
{
    grid_dependents_launch();
    const int pair = blockIdx.y >> 1;
    const bool is_v = blockIdx.y & 1;
    const int64_t src = __ldg(block_mapping + 2 * pair);
    const int64_t dst = __ldg(block_mapping + 2 * pair + 1);
    if (src < 0 || dst < 0 || src >= src_blocks || dst >= dst_blocks) {
        if (blockIdx.x == 0 && threadIdx.x == 0 && !is_v)
            record_error(err, PA_DEVERR_BLOCK_RANGE);
        return;
    }
    const uint4 *from = (is_v ? src_v : src_k) + src * block_vecs;
    uint4 *to = (is_v ? dst_v : dst_k) + dst * block_vecs;
    constexpr int U = 4;
    for (long long base = (long long)blockIdx.x * 256 * U; base < block_vecs;
         base += (long long)gridDim.x * 256 * U) {
        uint4 t[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long e = base + u * 256 + threadIdx.x;
            if (e < block_vecs)
                t[u] = from[e];
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long e = base + u * 256 + threadIdx.x;
            if (e < block_vecs)
                to[e] = t[u];
        }
    }
}

// ---------------------------------------------------------------------------
// gather_kv (debug): contiguous K/V of every sequence through its table.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
gather_kv_kernel(uint4 *k_out, uint4 *v_out, const uint4 *__restrict__ k_cache,
                 const uint4 *__restrict__ v_cache, const int32_t *__restrict__ block_tables,
                 const int32_t *__restrict__ seq_lens, int num_seqs, int num_kv_heads,
                 int row_vecs, int max_blocks, long long num_blocks, uint32_t *err)
{
    const int maxlen = max_blocks * kBlockSize;
    const long long total = (long long)num_seqs * num_kv_heads * maxlen * row_vecs;
    for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x < total;
         x += (long long)gridDim.x * blockDim.x) {
        const int vec = (int)(x % row_vecs);
        long long y = x / row_vecs;
        const int t = (int)(y % maxlen);
        y /= maxlen;
        const int kvh = (int)(y % num_kv_heads);
        const int s = (int)(y / num_kv_heads);
        int L = __ldg(seq_lens + s);
        if (L < 0 || L > maxlen) {
            if (t == 0 && vec == 0 && kvh == 0)
                record_error(err, PA_DEVERR_SEQLEN_RANGE);
            L = L < 0 ? 0 : maxlen;
        }
        if (t >= L)
            continue;
        const int phys = __ldg(block_tables + (long long)s * max_blocks + t / kBlockSize);
        if (phys < 0 || phys >= num_blocks) {
            if (t % kBlockSize == 0 && vec == 0)
                record_error(err, PA_DEVERR_TABLE_RANGE);
            continue;
        }
        const long long src = (((long long)phys * num_kv_heads + kvh) * kBlockSize + t % kBlockSize) *
                                  row_vecs + vec;
        k_out[x] = k_cache[src];
        v_out[x] = v_cache[src];
    }
}

// ---------------------------------------------------------------------------
// validate_tables: count table entries a decode would read that are outside
// the pool, and lengths outside [0, max_blocks * 16].
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
validate_tables_kernel(const int32_t *__restrict__ block_tables,
                       const int32_t *__restrict__ seq_lens, int num_seqs, int max_blocks,
                       int num_blocks, uint32_t *bad_count)
{
    const long long total = (long long)num_seqs * max_blocks;
    uint32_t bad = 0;
    for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x < total;
         x += (long long)gridDim.x * blockDim.x) {
        const int s = (int)(x / max_blocks), b = (int)(x % max_blocks);
        const int L = __ldg(seq_lens + s);
        if (b == 0 && (L < 0 || L > max_blocks * kBlockSize))
            ++bad;
        const int nb = (max(0, min(L, max_blocks * kBlockSize)) + kBlockSize - 1) / kBlockSize;
        if (b < nb) {
            const int e = __ldg(block_tables + x);
            if (e < 0 || e >= num_blocks)
                ++bad;
        }
    }
    if (bad)
        atomicAdd(bad_count, bad);
}

// ---------------------------------------------------------------------------
// Self-test of the bounded wait: an mbarrier expects bytes that no copy will
// deliver, so the wait must give up after limit_ns, record
// PA_DEVERR_TIMEOUT and let the kernel finish.  Nothing is in flight.
// ---------------------------------------------------------------------------
__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns, uint32_t *err)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_arrive_expect_tx(b, 16);      // 16 bytes that never arrive
    __syncthreads();
    if (!mbar_wait_bounded(b, 0, limit_ns) && threadIdx.x == 0)
        record_error(err, PA_DEVERR_TIMEOUT);
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
template <typename F>
static int resident_blocks(F *fn, int threads)
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, 0) != cudaSuccess || n < 1)
        n = 1;
    return n;
}

static int grid_for(long long work, int threads, int num_sms)
{
    long long g = (work + threads - 1) / threads;
    const long long cap = (long long)num_sms * 16;
    if (g > cap)
        g = cap;
    return (int)(g < 1 ? 1 : g);
}

cudaError_t launch_reshape_and_cache(const void *k_new, const void *v_new, void *k_cache,
                                     void *v_cache, const int64_t *slot_mapping, int num_tokens,
                                     int num_kv_heads, int head_dim, int num_blocks,
                                     uint32_t *err, int num_sms, cudaStream_t stream)
{
    const int row_shift = head_dim == 64 ? 3 : 4;           // 16-byte vectors per row, log2
    const long long total = (2LL * num_tokens * num_kv_heads) << row_shift;
    // one wave of resident blocks at most, looping; four vectors a thread
    // when that still gives every SM a block, else one (a decode step's few
    // tokens spread over more blocks)
    const long long slots = (long long)num_blocks * kBlockSize;
    const long long need4 = (total + 1023) / 1024, need1 = (total + 255) / 256;
    if (need4 >= num_sms) {
        static const int resident = resident_blocks(reshape_and_cache_kernel<4>, 256);
        const long long cap = (long long)num_sms * resident;
        reshape_and_cache_kernel<4><<<(int)(need4 < cap ? need4 : cap), 256, 0, stream>>>(
            static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new),
            static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), slot_mapping,
            num_tokens, num_kv_heads, row_shift, slots, err);
    } else {
        reshape_and_cache_kernel<1><<<(int)need1, 256, 0, stream>>>(
            static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new),
            static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), slot_mapping,
            num_tokens, num_kv_heads, row_shift, slots, err);
    }
    return cudaGetLastError();
}

cudaError_t launch_copy_blocks(void *dst_k, void *dst_v, const void *src_k, const void *src_v,
                               const int64_t *block_mapping, int num_pairs, int num_kv_heads,
                               int head_dim, long long src_blocks, long long dst_blocks,
                               uint32_t *err, cudaStream_t stream)
{
    const long long block_vecs = (long long)num_kv_heads * kBlockSize * head_dim * 2 / 16;
    const int gx = (int)((block_vecs + 256 * 4 - 1) / (256 * 4));
    for (int first = 0; first < num_pairs; first += 30000) {
        const int cnt = num_pairs - first < 30000 ? num_pairs - first : 30000;
        dim3 grid(gx, 2 * cnt);
        copy_blocks_kernel<<<grid, 256, 0, stream>>>(
            static_cast<uint4 *>(dst_k), static_cast<uint4 *>(dst_v),
            static_cast<const uint4 *>(src_k), static_cast<const uint4 *>(src_v),
            block_mapping + 2LL * first, cnt, block_vecs, src_blocks, dst_blocks, err);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

cudaError_t launch_gather_kv(void *k_out, void *v_out, const void *k_cache, const void *v_cache,
                             const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                             int num_kv_heads, int head_dim, int max_blocks, int num_blocks,
                             uint32_t *err, int num_sms, cudaStream_t stream)
{
    const int row_vecs = head_dim * 2 / 16;
    const long long total = (long long)num_seqs * num_kv_heads * max_blocks * kBlockSize * row_vecs;
    gather_kv_kernel<<<grid_for(total, 256, num_sms), 256, 0, stream>>>(
        static_cast<uint4 *>(k_out), static_cast<uint4 *>(v_out),
        static_cast<const uint4 *>(k_cache), static_cast<const uint4 *>(v_cache), block_tables,
        seq_lens, num_seqs, num_kv_heads, row_vecs, max_blocks, num_blocks, err);
    return cudaGetLastError();
}

cudaError_t launch_validate_tables(const int32_t *block_tables, const int32_t *seq_lens,
                                   int num_seqs, int max_blocks, int num_blocks,
                                   uint32_t *bad_count, int num_sms, cudaStream_t stream)
{
    const long long total = (long long)num_seqs * max_blocks;
    validate_tables_kernel<<<grid_for(total, 256, num_sms), 256, 0, stream>>>(
        block_tables, seq_lens, num_seqs, max_blocks, num_blocks, bad_count);
    return cudaGetLastError();
}

cudaError_t launch_bounded_wait_selftest(uint64_t limit_ns, uint32_t *err, cudaStream_t stream)
{
    bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
    return cudaGetLastError();
}

}  // namespace pa
