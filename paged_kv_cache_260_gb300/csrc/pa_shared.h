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
    const int32_t *seq_lens;       // [num_seqs]
    const void *k_new, *v_new;     // [num_seqs][num_kv_heads][head_dim], or null
    const int64_t *slot_mapping;   // [num_seqs], or null
    int num_seqs, group_size, prefix_tiles;
    int num_heads, num_kv_heads, head_dim, max_blocks;
    // The virtual batch, one decode: first nvb prefix sequences per group
    // (16 query columns (sample, head) per kv head, the group's first table
    // up to the prefix), then one suffix sequence per sequence (its heads in
    // the first G columns, its table past the prefix).
    int nvb, npre;                 // prefix sequences per group, in all
    int vmax_blocks;               // table row length of the virtual batch
    void *q_v;                     // [nv][num_kv_heads][16][head_dim]
    int32_t *tables_v;             // [nv][vmax_blocks]
    int32_t *lens_v;               // [nv]
    void *k_new_v, *v_new_v;       // [nv][num_kv_heads][head_dim] (append only)
    int64_t *slots_v;              // [nv] (append only; -1 for prefix sequences)
    uint32_t *err;                 // device error bits
    // the merge: partials [nv][num_kv_heads * 16] (m, l, o normalised), fp32
    const float *pm, *pl, *po;
    void *out;                     // [num_seqs][num_heads][head_dim]
};

cudaError_t launch_shared_prep(const SharedParams &p, int num_vseqs, cudaStream_t st);
cudaError_t launch_shared_merge(const SharedParams &p, bool bf16, cudaStream_t st);

}  // namespace pa
