// pa_shared.h -- what the host side of pa_decode_shared_prefix shares with
// its helper kernels (pa_shared.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pa {

struct SharedParams {
    // the batch: groups of group_size consecutive sequences share their first
    // prefix_tiles blocks
    int num_seqs, group_size, prefix_tiles;
    int num_heads, num_kv_heads, head_dim;
    uint32_t *err;                 // device error bits
    // the merge: the suffix partials [num_seqs][num_heads] (m, l, o
    // normalised, fp32), and the prefix partials of prefix_attn_kernel
    // [nchunks][num_groups * num_kv_heads][cols] (m, l; o with head_dim more)
    const float *pm, *pl, *po;
    const float *xm, *xl, *xo;
    // a suffix run r = (s, kv head h) that the decode's balanced split cut
    // has no row in pm/pl/po: cut_of_run[2r] >= 0 is the first worker c0 of
    // its pieces and cut_of_run[2r + 1] = 2 * last worker + (c0's piece in
    // its last slot); each piece is in a worker slot of sm/sl/so
    // ([2 * workers][G] rows)
    const int32_t *cut_of_run;
    const float *sm, *sl, *so;
    int nchunks, cols;             // key chunks of the prefix; group_size * G
    void *out;                     // [num_seqs][num_heads][head_dim]
};

// Attention of every query column (sample, head) of a group over the
// group's shared prefix, each prefix tile read once for all of them.
struct PrefixParams {
    const void *q;                 // [num_seqs][num_heads][head_dim]
    const int32_t *block_tables;   // [num_seqs][max_blocks]; a group's first row names the prefix
    int num_heads, num_kv_heads, max_blocks, num_blocks;
    int group_size, num_groups;
    int cols;                      // query columns of a (group, kv head): group_size * G
    int col_blocks;                // blocks of kPrefixCols columns per (group, kv head)
    int prefix_tiles, chunk_tiles, nchunks;
    float scale_log2;
    uint32_t *err;
    float *xm, *xl, *xo;           // partials [nchunks][num_groups * num_kv_heads][cols]
    // the suffix decode's lengths, written on the way: lens_v[s] =
    // seq_lens[s] - 16 prefix_tiles (0 and PA_DEVERR_SEQLEN_RANGE if shorter)
    const int32_t *seq_lens;
    int32_t *lens_v;
    int num_seqs;
};

constexpr int kPrefixCols = 64;    // query columns of one prefix thread block

cudaError_t launch_shared_merge(const SharedParams &p, bool bf16, cudaStream_t st);
// prefix_attn_kernel for the dtype and head size, launched with arguments
// (PrefixParams, CUtensorMap K pool, CUtensorMap V pool): a grid of
// nchunks * num_groups * num_kv_heads * col_blocks blocks
struct PrefixKernel {
    const void *fn;
    size_t smem;                   // dynamic shared memory a block
    int threads, blocks;
};
PrefixKernel prefix_kernel(const PrefixParams &p, bool bf16, int head_dim);

}  // namespace pa
