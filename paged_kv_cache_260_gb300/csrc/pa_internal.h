// pa_internal.h -- structures shared by the host dispatch and the kernels.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace pa {

constexpr int kBlockSize = 16;  // tokens per KV block

// How the (sequence, kv head) token runs are cut into work for the warps.
enum DecodeMode : int {
    kModeBalanced = 0,  // equal tile ranges per warp, merge of cut runs
    kModeFixed = 1,     // equal tile ranges, runs also cut into partitions, merge per partition
    kModeWhole = 2,     // no split: whole runs per warp
};

struct CutDesc;

struct DecodeParams {
    void *out;
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    const void *k_new;             // append: token s's K/V [num_seqs][Hkv][D], or null
    const void *v_new;
    const int64_t *slot_mapping;   // append: slot of position seq_lens[s] - 1, <0 = none
    float *ws_m;           // fixed mode, per partition: max of scaled scores (natural-log units)
    float *ws_l;           //   sum of exp(score - m)
    float *ws_o;           //   normalised partial output
    float *ws_sm;          // per worker slot (first / last piece): the same three results
    float *ws_sl;
    float *ws_so;
    CutDesc *ws_desc;      // per worker: the cut unit that starts in its range
    uint32_t *err;         // device error bits (PA_DEVERR_*)
    int num_seqs;
    int num_heads;
    int num_kv_heads;
    int max_blocks;        // block-table row length
    int num_blocks;        // pool size in blocks
    int mode;
    int part_tiles;        // fixed mode: tiles per partition
    int p_max;             // fixed mode: partitions per sequence (workspace stride)
    int min_tiles;         // least tiles given to one worker
    int workers;           // warps of the decode grid
    float scale_log2;      // scale * log2(e): scores are kept in base 2
};

// Kernels of one (dtype, head_dim) instantiation.  decode[0] is the wide
// variant (one block of many warps per SM); decode[1] a compact one used when
// the per-sequence arrays of a large batch leave too little shared memory.
struct KernelSet {
    const void *decode[2];
    int warps[2];            // warps (workers) per decode thread block
    size_t smem_fixed[2];    // dynamic shared memory excluding the per-sequence arrays
    const void *merge_cut;   // combines the pieces of cut units
    const void *merge_part;  // fixed mode: merges partitions into the output
};

// Per-sequence shared-memory arrays of the decode kernel: unit prefix
// [num_seqs + 1] and clamped lengths [num_seqs], int32 each.
inline size_t decode_smem_bytes(size_t smem_fixed, int num_seqs)
{
    return smem_fixed + sizeof(int32_t) * (2 * (size_t)num_seqs + 1);
}

constexpr int kMaxSeqs = 8192;        // per-sequence arrays live in shared memory
constexpr int kMaxWarpsPerSM = 16;    // decode workers <= SMs * this (workspace sizing)
constexpr int kMinTiles = 2;          // split modes: least tiles per worker (warp)

bool decode_kernels_f16(int head_dim, int group, KernelSet *ks);
bool decode_kernels_bf16(int head_dim, int group, KernelSet *ks);

}  // namespace pa
