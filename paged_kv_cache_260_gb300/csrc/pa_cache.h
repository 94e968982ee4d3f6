// pa_cache.h -- launchers of the pool-maintenance kernels (host side).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

cudaError_t launch_reshape_and_cache(const void *k_new, const void *v_new, void *k_cache,
                                     void *v_cache, const int64_t *slot_mapping, int num_tokens,
                                     int num_kv_heads, int head_dim, int num_blocks,
                                     uint32_t *err, int num_sms, cudaStream_t stream);

cudaError_t launch_copy_blocks(void *dst_k, void *dst_v, const void *src_k, const void *src_v,
                               const int64_t *block_mapping, int num_pairs, int num_kv_heads,
                               int head_dim, long long src_blocks, long long dst_blocks,
                               uint32_t *err, cudaStream_t stream);

cudaError_t launch_gather_kv(void *k_out, void *v_out, const void *k_cache, const void *v_cache,
                             const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                             int num_kv_heads, int head_dim, int max_blocks, int num_blocks,
                             uint32_t *err, int num_sms, cudaStream_t stream);

cudaError_t launch_validate_tables(const int32_t *block_tables, const int32_t *seq_lens,
                                   int num_seqs, int max_blocks, int num_blocks,
                                   uint32_t *bad_count, int num_sms, cudaStream_t stream);

cudaError_t launch_bounded_wait_selftest(uint64_t limit_ns, uint32_t *err, cudaStream_t stream);

}  // namespace pa
