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
    int32_t *ws_pre;       // large batches: unit prefix [num_seqs + 1] in the workspace, or null
    int32_t *ws_lens;      //   clamped lengths [num_seqs] (null: all three in shared memory)
    uint8_t *ws_share;     //   and first-block-shared flags [num_seqs]
    int32_t *ws_blk;       //   the prep kernels' per-block unit count and any-flag
                           //   [ceil(num_seqs / kPrepSeqs)][2]
    float *out_m;          // partial-output mode (non-null): each (sequence, query head)'s
    float *out_l;          //   m, l and normalised o go to row s * num_heads + h of these
    float *out_o;          //   [num_seqs][num_heads](x head_dim) fp32 arrays instead of `out`
    int32_t *cut_of_run;   // partial-output mode, balanced split (or null): per run
                           //   r = s * num_kv_heads + h two ints, [2r] = -1 if the run is
                           //   empty or one worker covered it whole, else the first worker
                           //   c0 of its pieces, and [2r + 1] = 2 * last worker + (c0's
                           //   piece in its last slot); the caller then folds the pieces
                           //   itself and no merge_cut runs
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

// Kernels of one (dtype, head_dim, query columns) instantiation.
struct KernelSet {
    const void *decode;      // one thread block per SM of `warps` independent warps
    const void *decode_partial;  // the same writing fp32 partial results (16 columns only)
    int warps;
    size_t smem_fixed;       // dynamic shared memory excluding the per-sequence arrays
    const void *prep;        // large batches: build the per-sequence arrays in the workspace,
    const void *prep_fix;    //   block by block, then add the earlier blocks' unit counts
    const void *merge_cut;   // combines the pieces of cut units
    const void *merge_part;  // fixed mode: merges partitions into the output
};

// Per-sequence shared-memory arrays of the decode kernel: unit prefix
// [num_seqs + 1] and clamped lengths [num_seqs], int32 each, then one
// first-block-shared flag byte per sequence.
inline size_t decode_smem_bytes(size_t smem_fixed, int num_seqs)
{
    return smem_fixed + sizeof(int32_t) * (2 * (size_t)num_seqs + 1) + (size_t)num_seqs;
}

// Batches up to this size keep the per-sequence arrays in each decode block's
// shared memory (every variant fits them under the 227 KiB limit); larger
// ones have them built once in the workspace by the prep kernel.
constexpr int kSeqsInSmem = 2048;
constexpr int kPrepThreads = 256;
constexpr int kPrepSeqs = 4 * kPrepThreads;   // sequences a prep block builds
constexpr int kMaxWarpsPerSM = 16;    // decode workers <= SMs * this (workspace sizing)
constexpr int kMinTiles = 2;          // split modes: least tiles per worker (warp)
// Balanced mode falls back to whole runs when every table is at most this
// many blocks wide and the runs number at most kWholeRunsPerSM per SM.
constexpr int kWholeMaxBlocks = 8;
constexpr int kWholeRunsPerSM = 4;
constexpr int kMaxGroup = 16;         // query heads per kv head: two 8-column tiles

bool decode_kernels_f16(int head_dim, KernelSet *ks);       // groups 1..8
bool decode_kernels_bf16(int head_dim, KernelSet *ks);
bool decode_kernels_f16_g16(int head_dim, KernelSet *ks);   // groups 9..16
bool decode_kernels_bf16_g16(int head_dim, KernelSet *ks);

}  // namespace pa
