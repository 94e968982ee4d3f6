// pa_internal.h -- structures shared by the host dispatch and the kernels.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace pa {

constexpr int kBlockSize = 16;  // tokens per KV block

// How the (sequence, kv head) token runs are cut into work for thread blocks.
enum DecodeMode : int {
    kModeBalanced = 0,  // equal tile ranges per thread block, merge of cut runs
    kModeFixed = 1,     // fixed partitions of part_tiles tiles, merge of partitions
    kModeWhole = 2,     // no split: one thread block per run
};

struct DecodeParams {
    void *out;
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    float *ws_m;           // partial max of scaled scores (natural-log units)
    float *ws_l;           // partial sum of exp(score - m)
    float *ws_o;           // partial normalised output
    int32_t *ws_prefix;    // balanced mode: per-sequence tile prefix, for the merge
    uint32_t *err;         // device error bits (PA_DEVERR_*)
    int num_seqs;
    int num_heads;
    int num_kv_heads;
    int max_blocks;        // block-table row length
    int num_blocks;        // pool size in blocks
    int mode;
    int part_tiles;        // fixed mode: tiles per partition
    int p_max;             // fixed mode: partitions per sequence (workspace stride)
    int min_tiles;         // balanced mode: least tiles given to one thread block
    int grid;              // decode grid size (the merge needs it)
    float scale_log2;      // scale * log2(e): scores are kept in base 2
};

// Kernels of one (dtype, head_dim, group) instantiation.
struct KernelSet {
    const void *decode;
    const void *merge;
    int warps;         // warps per decode thread block
    int stages;        // copy stages per warp
    size_t smem_fixed; // dynamic shared memory excluding the per-sequence arrays
};

// Per-sequence shared-memory arrays of the decode kernel: unit prefix
// [num_seqs + 1] and clamped lengths [num_seqs], int32 each.
inline size_t decode_smem_bytes(const KernelSet &ks, int num_seqs)
{
    return ks.smem_fixed + sizeof(int32_t) * (2 * (size_t)num_seqs + 1);
}

constexpr int kMaxSeqs = 8192;        // per-sequence arrays live in shared memory
constexpr int kMaxBlocksPerSM = 4;    // decode grid <= SMs * this (workspace sizing)
constexpr int kMinTiles = 8;          // balanced mode: least tiles per thread block

bool decode_kernels_f16(int head_dim, int group, KernelSet *ks);
bool decode_kernels_bf16(int head_dim, int group, KernelSet *ks);

}  // namespace pa
