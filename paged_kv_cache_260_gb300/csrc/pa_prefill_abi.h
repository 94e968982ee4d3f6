// pa_prefill_abi.h -- what the host side of pa_prefill shares with the
// prefill kernels: their parameters, the launch descriptor and the tile
// sizes.  Kept apart from the decode's declarations.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace pa {

// Chunked prefill: the newest chunk_s = query_start[s+1] - query_start[s]
// tokens of sequence s (already in the pool) attend causally to positions
// [0, own position] of the sequence.
struct PrefillParams {
    void *out;                     // [total_q][num_heads][head_dim]
    const void *q;                 // [total_q][num_heads][head_dim]
    const int32_t *block_tables;
    const int32_t *seq_lens;
    const int32_t *query_start;    // [num_seqs + 1]
    uint32_t *err;
    int num_seqs;
    int num_heads;
    int num_kv_heads;
    int max_blocks;
    int num_blocks;
    int q_ranks;                   // query tiles per (sequence, kv head) in the grid
    float scale_log2;
    // optional work order (a planning kernel writes it): a list of
    // (sequence << 16 | query tile) pairs, *plan_count of them, heaviest
    // first; null: the grid is walked as (query tile from the end, sequence,
    // kv head).  Block b takes pair plan[b / num_kv_heads] and kv head
    // b % num_kv_heads, except when *plan_by_seq is set (the pairs are then
    // grouped by sequence, sequence s owning plan[seq_start[s] ..
    // seq_start[s] + seq_nq[s])): there the blocks of a sequence take its
    // kv heads one after the other, each head with all of the sequence's
    // query tiles, so that the blocks running at one time read few heads'
    // K/V and no wave spans two sequences' whole K/V.
    const uint32_t *plan;
    const int *plan_count;
    const int *plan_by_seq;
    const int32_t *plan_seq_start;
    const int32_t *plan_seq_nq;
    // blocks in one wave (the SM count): with a work order, block b warms
    // L2 with the query rows of block b + wave, which starts about when a
    // block of this wave ends
    int wave;
};

struct PrefillKernel {
    const void *fn;
    int threads;
    size_t smem;
    const void *plan_fn;           // prefill_plan_kernel: (PrefillParams, tokens per block,
                                   // keys per tile, uint32_t *plan, int *count,
                                   // long long K+V bytes per token, long long L2 bytes,
                                   // int *by_seq, int32_t *seq_start, int32_t *seq_nq)
};

bool prefill_kernel(int dtype, int head_dim, PrefillKernel *k);
constexpr int kPrefillRows = 128;   // (token, head) rows of one prefill query tile
constexpr int kPrefillTiles = 2;    // query tiles of one prefill thread block
constexpr int kPrefillKeys = 128;   // keys per prefill key tile

}  // namespace pa
