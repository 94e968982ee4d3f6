// pa_shared.cu -- the two helper kernels of pa_decode_shared_prefix.
//
// Parallel samples of one prompt share the prompt's KV blocks by reference
// (block sharing with copy-on-write, section 系统实现要点 of the vLLM reading
// notes; the page-sharing row of its OS-paging table).  Decoding each sample
// on its own streams the shared blocks once per sample.  pa_decode_shared_prefix
// instead decodes the shared prefix once per group of samples, as "virtual
// sequences" that each hold up to 16 query columns (sample, head) of one
// group and kv head and read the prefix through the group's first table.
// The samples' own suffixes are further virtual sequences of the same
// decode launch, and each (sample, head)'s two partial results are combined
// with the log-sum-exp rule (the same split-K merge the decode uses,
// FlashDecoding in the ICML tutorial notes, section "内核优化").
//
//  * shared_prep_kernel gathers the virtual batch of one decode: the prefix
//    sequences (query columns, the group's prefix table row) and the suffix
//    sequences (each sample's heads, its table past the prefix, its new
//    token).
//  * shared_merge_kernel combines each (sample, head)'s prefix partial with
//    its suffix partial into the output.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "pa_shared.h"
#include "pagedattn.h"

namespace pa {
namespace {

// Programmatic dependent launch: wait for the preceding grid, let the next
// be scheduled early.
__device__ __forceinline__ void grid_dependency_wait_()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dependents_launch_()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

constexpr int kCols = 16;   // query columns of a virtual sequence per kv head

// Block (v, kv head) fills virtual sequence v for that kv head.
//  * v < npre, a prefix sequence of group g = v / nvb, b = v % nvb: column c'
//    holds the group's column c = 16 b + c' (sample c / G, head c % G), zero
//    past the group's columns; its table is the group's first table up to
//    the prefix, its length the prefix.
//  * v >= npre, the suffix of sequence s = v - npre: columns 0..G-1 hold its
//    heads; its table is its own past the prefix, its length what lies past
//    the prefix, and it carries the sequence's new token.
__global__ void __launch_bounds__(256) shared_prep_kernel(const SharedParams p)
{
    grid_dependents_launch_();
    grid_dependency_wait_();
    const int v = blockIdx.x, h = blockIdx.y;
    const int G = p.num_heads / p.num_kv_heads;
    const int vec = p.head_dim / 8;                  // 16-byte vectors per query row
    const uint4 *q = static_cast<const uint4 *>(p.q);
    uint4 *qv = static_cast<uint4 *>(p.q_v);
    const bool pre = v < p.npre;
    const int g = pre ? v / p.nvb : 0, b = pre ? v - g * p.nvb : 0, s = pre ? 0 : v - p.npre;
    for (int i = threadIdx.x; i < kCols * vec; i += blockDim.x) {
        const int cc = i / vec, x = i - cc * vec;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (pre) {
            const int c = b * kCols + cc;
            if (c < p.group_size * G)
                val = q[((size_t)(g * p.group_size + c / G) * p.num_heads + h * G + c % G) * vec + x];
        } else if (cc < G) {
            val = q[((size_t)s * p.num_heads + h * G + cc) * vec + x];
        }
        qv[(((size_t)v * p.num_kv_heads + h) * kCols + cc) * vec + x] = val;
    }
    if (!pre && p.k_new_v) {
        const uint4 *kn = static_cast<const uint4 *>(p.k_new);
        const uint4 *vn = static_cast<const uint4 *>(p.v_new);
        const size_t src = ((size_t)s * p.num_kv_heads + h) * vec, dst = ((size_t)v * p.num_kv_heads + h) * vec;
        for (int x = threadIdx.x; x < vec; x += blockDim.x) {
            static_cast<uint4 *>(p.k_new_v)[dst + x] = kn[src + x];
            static_cast<uint4 *>(p.v_new_v)[dst + x] = vn[src + x];
        }
    }
    if (h != 0)
        return;
    int32_t *row = p.tables_v + (size_t)v * p.vmax_blocks;
    if (pre) {
        const int32_t *src = p.block_tables + (size_t)g * p.group_size * p.max_blocks;
        for (int t = threadIdx.x; t < p.vmax_blocks; t += blockDim.x)
            row[t] = t < p.prefix_tiles ? src[t] : 0;
        if (threadIdx.x == 0) {
            p.lens_v[v] = p.prefix_tiles * 16;
            if (p.slots_v)
                p.slots_v[v] = -1;
        }
        return;
    }
    const int32_t *src = p.block_tables + (size_t)s * p.max_blocks + p.prefix_tiles;
    const int rest = p.max_blocks - p.prefix_tiles;
    for (int t = threadIdx.x; t < p.vmax_blocks; t += blockDim.x)
        row[t] = t < rest ? src[t] : 0;
    if (threadIdx.x == 0) {
        int L = p.seq_lens[s] - p.prefix_tiles * 16;
        if (L < 0) {                                 // shorter than the shared prefix
            if (p.err)
                atomicOr(p.err, PA_DEVERR_SEQLEN_RANGE);
            L = 0;
        }
        p.lens_v[v] = L;
        if (p.slots_v)
            p.slots_v[v] = p.slot_mapping[s];
    }
}

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x)
{
    return __float2bfloat16_rn(x);
}

// One warp per (sample, query head):
//     M = max(m_1, m_2), w_i = l_i exp(m_i - M), out = (w_1 o_1 + w_2 o_2) / (w_1 + w_2)
// over the prefix partial (its prefix sequence's column) and the suffix
// partial (its suffix sequence's column).
template <typename T>
__global__ void __launch_bounds__(256) shared_merge_kernel(const SharedParams p)
{
    grid_dependents_launch_();
    grid_dependency_wait_();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int rows = p.num_seqs * p.num_heads;
    if (warp >= rows)
        return;
    const int s = warp / p.num_heads, hq = warp - s * p.num_heads;
    const int G = p.num_heads / p.num_kv_heads;
    const int g = s / p.group_size, smp = s - g * p.group_size;
    const int h = hq / G, c = smp * G + hq % G;
    const size_t prow = ((size_t)(g * p.nvb + c / kCols) * p.num_kv_heads + h) * kCols + c % kCols;
    const size_t srow = ((size_t)(p.npre + s) * p.num_kv_heads + h) * kCols + hq % G;
    const float m1 = p.pm[prow], l1 = p.pl[prow];
    const float m2 = p.pm[srow], l2 = p.pl[srow];
    const float M = fmaxf(m1, m2);
    const float w1 = l1 > 0.f ? l1 * expf(m1 - M) : 0.f;
    const float w2 = l2 > 0.f ? l2 * expf(m2 - M) : 0.f;
    const float inv = w1 + w2 > 0.f ? 1.f / (w1 + w2) : 0.f;
    T *out = static_cast<T *>(p.out) + (size_t)warp * p.head_dim;
    for (int d = lane; d < p.head_dim; d += 32) {
        const float o1 = w1 > 0.f ? p.po[prow * p.head_dim + d] : 0.f;
        const float o2 = w2 > 0.f ? p.po[srow * p.head_dim + d] : 0.f;
        out[d] = from_f<T>((w1 * o1 + w2 * o2) * inv);
    }
}

}  // namespace

namespace {
cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, cudaStream_t st, const SharedParams &p)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<SharedParams *>(&p)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}
}  // namespace

// Both are programmatic dependent launches: scheduled while the preceding
// kernel drains, touching no global memory before it has completed.
cudaError_t launch_shared_prep(const SharedParams &p, int num_vseqs, cudaStream_t st)
{
    return launch_pdl(reinterpret_cast<const void *>(&shared_prep_kernel),
                      dim3(num_vseqs, p.num_kv_heads), dim3(256), st, p);
}

cudaError_t launch_shared_merge(const SharedParams &p, bool bf16, cudaStream_t st)
{
    const int rows = p.num_seqs * p.num_heads;
    const dim3 grid((rows + 7) / 8);
    return bf16 ? launch_pdl(reinterpret_cast<const void *>(&shared_merge_kernel<__nv_bfloat16>),
                             grid, dim3(256), st, p)
                : launch_pdl(reinterpret_cast<const void *>(&shared_merge_kernel<__half>), grid,
                             dim3(256), st, p);
}

}  // namespace pa
