// pa_shared.h -- what the host side of pa_decode_shared_prefix shares with
// its helper kernels (pa_shared.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pa {

struct SharedParams {
    // the batch: groups of group_size consecutive sequences share their first
    // prefix_tiles blocks
    const void *q;                 // [num_seqs][num_heads][head_dim]
    const int32_t *block_tables;   // [num_seqs][max_blocks]
    int num_seqs, group_size, prefix_tiles;
    int num_heads, num_kv_heads, head_dim, max_blocks;
    // the virtual batch: nvb virtual sequences per group, cv query columns
    // (sample, head) per kv head each
    int nvb, cv;
    void *q_v;                     // [groups * nvb][num_kv_heads][cv][head_dim]
    int32_t *tables_v;             // [groups * nvb][prefix_tiles]
    int32_t *lens_v;               // [groups * nvb]
    // the merge: prefix partials [groups * nvb][num_kv_heads * cv] and suffix
    // partials [num_seqs][num_heads] (m, l, o normalised), fp32
    const float *pm, *pl, *po;
    const float *sm, *sl, *so;
    void *out;                     // [num_seqs][num_heads][head_dim]
};

cudaError_t launch_shared_prep(const SharedParams &p, int num_vseqs, cudaStream_t st);
cudaError_t launch_shared_merge(const SharedParams &p, bool bf16, cudaStream_t st);

}  // namespace pa
