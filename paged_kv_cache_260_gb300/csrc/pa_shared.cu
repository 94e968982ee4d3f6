// pa_shared.cu -- the two helper kernels of pa_decode_shared_prefix.
//
// Parallel samples of one prompt share the prompt's KV blocks by reference
// (block sharing with copy-on-write, section 系统实现要点 of the vLLM reading
// notes; the page-sharing row of its OS-paging table).  Decoding each sample
// on its own streams the shared blocks once per sample.  pa_decode_shared_prefix
// instead decodes the shared prefix once per group of samples, as a batch of
// "virtual sequences": each holds up to 16 query columns (sample, head) of
// one group and kv head and reads the prefix through the group's first
// table.  The samples' own suffixes are a second decode, and the two partial
// results are combined with the log-sum-exp rule (the same split-K merge the
// decode uses, FlashDecoding in the ICML tutorial notes, section "内核优化").
//
//  * shared_prep_kernel gathers the virtual batch: query columns, the group's
//    prefix table row, the prefix length.
//  * shared_merge_kernel combines each (sample, head)'s prefix partial with
//    its suffix partial into the output.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "pa_shared.h"

namespace pa {
namespace {

// Block (vseq, kv head): columns c' = 0..cv-1 of virtual sequence vseq are
// the group's columns c = b * cv + c' (sample c / G, head c % G of the kv
// head); columns past the group's are zero.  Block (vseq, 0) also writes the
// virtual table row and length.
__global__ void __launch_bounds__(256) shared_prep_kernel(const SharedParams p)
{
    const int vseq = blockIdx.x, h = blockIdx.y;
    const int g = vseq / p.nvb, b = vseq - g * p.nvb;
    const int G = p.num_heads / p.num_kv_heads;
    const int cols = p.group_size * G;
    const int vec = p.head_dim / 8;                  // 16-byte vectors per query row
    const uint4 *q = static_cast<const uint4 *>(p.q);
    uint4 *qv = static_cast<uint4 *>(p.q_v);
    for (int i = threadIdx.x; i < p.cv * vec; i += blockDim.x) {
        const int cc = i / vec, x = i - cc * vec;
        const int c = b * p.cv + cc;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (c < cols) {
            const int s = g * p.group_size + c / G, hq = h * G + c % G;
            val = q[((size_t)s * p.num_heads + hq) * vec + x];
        }
        qv[(((size_t)vseq * p.num_kv_heads + h) * p.cv + cc) * vec + x] = val;
    }
    if (h == 0) {
        const int32_t *row = p.block_tables + (size_t)g * p.group_size * p.max_blocks;
        for (int t = threadIdx.x; t < p.prefix_tiles; t += blockDim.x)
            p.tables_v[(size_t)vseq * p.prefix_tiles + t] = row[t];
        if (threadIdx.x == 0)
            p.lens_v[vseq] = p.prefix_tiles * 16;
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
// over the prefix partial (from its virtual sequence's column) and the
// suffix partial.
template <typename T>
__global__ void __launch_bounds__(256) shared_merge_kernel(const SharedParams p)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int rows = p.num_seqs * p.num_heads;
    if (warp >= rows)
        return;
    const int s = warp / p.num_heads, hq = warp - s * p.num_heads;
    const int G = p.num_heads / p.num_kv_heads;
    const int g = s / p.group_size, smp = s - g * p.group_size;
    const int h = hq / G, c = smp * G + hq % G;
    const int vseq = g * p.nvb + c / p.cv;
    const size_t prow = ((size_t)vseq * p.num_kv_heads + h) * p.cv + c % p.cv;
    const size_t srow = (size_t)warp;
    const float m1 = p.pm[prow], l1 = p.pl[prow];
    const float m2 = p.sm[srow], l2 = p.sl[srow];
    const float M = fmaxf(m1, m2);
    const float w1 = l1 > 0.f ? l1 * expf(m1 - M) : 0.f;
    const float w2 = l2 > 0.f ? l2 * expf(m2 - M) : 0.f;
    const float inv = w1 + w2 > 0.f ? 1.f / (w1 + w2) : 0.f;
    T *out = static_cast<T *>(p.out) + srow * p.head_dim;
    for (int d = lane; d < p.head_dim; d += 32) {
        const float o1 = w1 > 0.f ? p.po[prow * p.head_dim + d] : 0.f;
        const float o2 = w2 > 0.f ? p.so[srow * p.head_dim + d] : 0.f;
        out[d] = from_f<T>((w1 * o1 + w2 * o2) * inv);
    }
}

}  // namespace

cudaError_t launch_shared_prep(const SharedParams &p, int num_vseqs, cudaStream_t st)
{
    shared_prep_kernel<<<dim3(num_vseqs, p.num_kv_heads), 256, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_shared_merge(const SharedParams &p, bool bf16, cudaStream_t st)
{
    const int rows = p.num_seqs * p.num_heads;
    const int blocks = (rows + 7) / 8;
    if (bf16)
        shared_merge_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(p);
    else
        shared_merge_kernel<__half><<<blocks, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace pa
