// pa_shared.cu -- the helper kernels of pa_decode_shared_prefix.
//
// Parallel samples of one prompt share the prompt's KV blocks by reference
// (block sharing with copy-on-write, section 系统实现要点 of the vLLM reading
// notes; the page-sharing row of its OS-paging table).  Decoding each sample
// on its own streams the shared blocks once per sample.  pa_decode_shared_prefix
// instead attends every query column (sample, head) of a group over the
// shared prefix at once, reading each prefix block once (prefix_attn_kernel,
// pa_prefix.cu), decodes the samples' own suffixes (their tables past the
// prefix) in one decode launch, and combines each (sample, head)'s partial results with
// the log-sum-exp rule (the same split-K merge the decode uses,
// FlashDecoding in the ICML tutorial notes, section "内核优化").
//
//  * shared_merge_kernel combines each (sample, head)'s prefix partials (one
//    per key chunk) with its suffix partial -- or, where the suffix decode's
//    balanced split cut the run, with the run's pieces -- into the output.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_schedule.cuh"
#include "pa_shared.h"
#include "pagedattn.h"

namespace pa {
namespace {

// One warp per (sample, query head), over its partials (m_i, l_i, o_i) --
// the prefix's key chunks, then the suffix (one row, or the pieces of a cut
// run in the decode's worker slots):
//     M = max_i m_i,  w_i = l_i exp(m_i - M),  out = sum_i w_i o_i / sum_i w_i
// Lane i reads partial i's m and l (32 at a time), so the weights need one
// warp reduction, and the o rows are then summed eight at a time with their
// loads in flight together.
template <typename T>
__global__ void __launch_bounds__(256) shared_merge_kernel(const SharedParams p)
{
    grid_dependents_launch();
    grid_dependency_wait();
    constexpr uint32_t FULL = 0xffffffffu;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int rows = p.num_seqs * p.num_heads;
    if (warp >= rows)
        return;
    const int s = warp / p.num_heads, hq = warp - s * p.num_heads;
    const int G = p.num_heads / p.num_kv_heads;
    const int g = s / p.group_size, smp = s - g * p.group_size;
    const int h = hq / G, c = smp * G + hq % G;
    const size_t cstride = (size_t)(p.num_seqs / p.group_size) * p.num_kv_heads * p.cols;
    const size_t xrow = ((size_t)g * p.num_kv_heads + h) * p.cols + c;   // chunk 0
    // the prefix chunks' m and l (partial `lane` of the first 32), loaded
    // while the suffix's record is looked up
    const int nx = p.nchunks;
    float mr = -INFINITY, lr = 0.f;
    if (lane < nx) {
        mr = p.xm[xrow + (size_t)lane * cstride];
        lr = p.xl[xrow + (size_t)lane * cstride];
    }
    // the suffix: row `warp` of pm/pl/po, or the pieces of a cut run
    const int2 cut = __ldcg(reinterpret_cast<const int2 *>(p.cut_of_run) +
                            (size_t)s * p.num_kv_heads + h);
    const int c0 = cut.x;
    const bool c0_last = cut.y & 1;
    const int nsuf = c0 >= 0 ? (cut.y >> 1) - c0 + 1 : 1;
    const float *sm = c0 >= 0 ? p.sm : p.pm;
    const float *sl = c0 >= 0 ? p.sl : p.pl;
    const float *so = c0 >= 0 ? p.so : p.po;
    const int np = nx + nsuf;                        // partials nx.. are the suffix's
    auto row_of = [&](int i) -> size_t {
        if (i < nx)
            return xrow + (size_t)i * cstride;
        if (c0 < 0)
            return (size_t)warp;
        return (size_t)cut_piece_slot(c0 + (i - nx), c0, c0_last) * G + hq % G;
    };
    auto m_of = [&](int i) { return i < nx ? p.xm[row_of(i)] : __ldcg(sm + row_of(i)); };
    auto l_of = [&](int i) { return i < nx ? p.xl[row_of(i)] : __ldcg(sl + row_of(i)); };
    auto o_of = [&](int i) { return (i < nx ? p.xo : so) + row_of(i) * p.head_dim; };
    if (lane >= nx && lane < np) {
        mr = m_of(lane);
        lr = l_of(lane);
    }
    // M over the non-empty partials
    float M = lr > 0.f ? mr : -INFINITY;
    for (int i = 32 + lane; i < np; i += 32) {
        if (l_of(i) > 0.f)
            M = fmaxf(M, m_of(i));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(FULL, M, off));
    constexpr int V = 4;                             // channels a lane, head_dim <= 128
    float W = 0.f, acc[V] = {0.f, 0.f, 0.f, 0.f};
    for (int base = 0; base < np; base += 32) {
        const int i = base + lane;
        float w = 0.f;
        if (i < np) {
            const float l = base == 0 ? lr : l_of(i);
            const float m = base == 0 ? mr : m_of(i);
            w = l > 0.f ? l * expf(m - M) : 0.f;     // an empty partial weighs nothing
        }
        const int cnt = min(32, np - base);
        for (int k0 = 0; k0 < cnt; k0 += 8) {
            // eight rows' loads in flight at once; every row is written by
            // the call, and an empty one is dropped by its weight below
            float ov[8][V];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (k0 + u < cnt) {
                    const float *o = o_of(base + k0 + u);
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        const int d = lane + 32 * v;
                        ov[u][v] = d < p.head_dim ? o[d] : 0.f;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (k0 + u < cnt) {
                    const float wk = __shfl_sync(FULL, w, k0 + u);
                    W += wk;
#pragma unroll
                    for (int v = 0; v < V; ++v)
                        acc[v] += wk > 0.f ? wk * ov[u][v] : 0.f;
                }
            }
        }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    T *out = static_cast<T *>(p.out) + (size_t)warp * p.head_dim;
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int d = lane + 32 * v;
        if (d < p.head_dim)
            out[d] = Elem<T>::from_f(acc[v] * inv);
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
