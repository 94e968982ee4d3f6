// pa_noalloc.cu -- pa_decode_noalloc: paged decode attention for callers that
// cannot allocate device memory.
//
// pa_decode wants a caller-owned workspace for its split-K partial results.
// Some callers have no way to provide one: an engine that hands (nearly) all
// free HBM to its KV block pool at start-up and allows no allocation
// afterwards, a plugin whose host framework passes only inputs and outputs,
// or code that runs where cudaMalloc is not allowed.  This entry point keeps
// the scratch in a fixed, file-scope device array instead, so it calls no
// cudaMalloc, cudaFree or allocating library routine.
//
// The array is loaded with the library's device code: every GPU that loads
// the library holds kNoAllocScratchBytes of it until the process exits.
#include <atomic>
#include <mutex>
#include <stdint.h>

#include "pa_internal.h"
#include "pagedattn.h"

namespace pa {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)PA_NOALLOC_SCRATCH_BYTES;

// Shared by every call on a device; holds whatever the last call left there.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
std::atomic<void *> g_noalloc_ptr[kMaxDevices];   // device address of the array, per device

// The array's device address on the current device.  The array's name is
// only a host-side stand-in, so the first call on a device looks the real
// address up (with that device current) under a lock; later calls read the
// cached pointer without one.
int scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return PA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return PA_ERR_UNSUPPORTED;
    void *p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        p = g_noalloc_ptr[dev].load(std::memory_order_relaxed);
        if (!p) {
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
                return PA_ERR_CUDA;
            g_noalloc_ptr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" int pa_decode_noalloc(void *out, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *block_tables,
                                 const int32_t *seq_lens, int num_seqs, int num_heads,
                                 int num_kv_heads, int head_dim, int block_size,
                                 int max_blocks_per_seq, int num_blocks, float scale, int dtype,
                                 void *stream)
{
    // The balanced split's scratch never needs clearing: every call writes
    // each worker's cut descriptor and every partial row before reading it.
    // An empty batch needs no scratch; pa_decode still checks its arguments.
    const size_t need = pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                                 max_blocks_per_seq, 0);
    if (need > pa::kNoAllocScratchBytes)
        return PA_ERR_WORKSPACE;
    void *scratch = nullptr;
    const int rc = pa::scratch_address(&scratch);
    if (rc != PA_OK)
        return rc;
    return pa_decode(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_heads,
                     num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale,
                     dtype, 0, scratch, pa::kNoAllocScratchBytes, stream);
}
