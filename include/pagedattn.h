/*
 * pagedattn.h -- C ABI of the GB300 (sm_103a) paged-KV-cache kernels.
 *
 * The KV cache lives in a pool of fixed 16-token blocks allocated once by the
 * caller; each sequence reaches its blocks through a block table (logical
 * block -> physical block), so attention reads K/V indirectly, exactly as an
 * MMU maps pages to frames ("PagedAttention：vLLM 系统论文" reading notes,
 * section 核心思想, block-pool figure and the OS-paging table; default block
 * of 16 tokens also in the vLLM deep notes, section "PagedAttention：操作系统
 * 启发的设计").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All pointers are DEVICE pointers, owned by the caller, 16-byte aligned.
 *    The library never allocates, frees or synchronises; every call only
 *    enqueues kernels on `stream` (a cudaStream_t passed as void*; NULL is the
 *    legacy default stream) and returns.
 *  - dtype: PA_DTYPE_F16 or PA_DTYPE_BF16, the type of q, out and both pools.
 *    Accumulation is fp32.
 *  - Pool layout ("HND"): k_cache, v_cache = [num_blocks][num_kv_heads]
 *    [block_size][head_dim], row-major.  Token t of sequence s lives in
 *    physical block block_tables[s][t / block_size] at offset
 *    t % block_size; slot numbers are block * block_size + offset.
 *  - block_size must be 16; head_dim 64 or 128; num_heads a multiple of
 *    num_kv_heads with a group G = num_heads / num_kv_heads of 1..16.  Query
 *    head h reads kv head h / G (grouped-query attention: several query heads
 *    share one K/V head, ICML tutorial notes, section "Attention 简化与 KV Cache
 *    优化").
 *  - Every call returns a pa_status.  Scalars and pointers are checked on the
 *    host before anything is enqueued.  Device arrays are not read on the
 *    host; kernels bounds-check every block id, slot and length they use,
 *    skip the offending access and record a PA_DEVERR_* bit that
 *    pa_get_device_error() returns.  No kernel traps.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PAGEDATTN_VERSION 1

enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or count */
    PA_ERR_UNSUPPORTED = 2,   /* head_dim, block_size, group or dtype not built */
    PA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
    PA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    PA_ERR_DEVICE = 5         /* a kernel recorded an error (see pa_get_device_error) */
};

enum pa_dtype { PA_DTYPE_F16 = 0, PA_DTYPE_BF16 = 1 };

/* bits recorded by kernels; read and cleared with pa_get_device_error() */
#define PA_DEVERR_SLOT_RANGE   0x1u  /* reshape_and_cache: slot >= num_blocks*block_size */
#define PA_DEVERR_BLOCK_RANGE  0x2u  /* copy_blocks: src or dst outside [0, num_blocks) */
#define PA_DEVERR_TABLE_RANGE  0x4u  /* decode/gather: table entry outside [0, num_blocks) */
#define PA_DEVERR_SEQLEN_RANGE 0x8u  /* seq_len < 0 or > max_blocks_per_seq*block_size */
#define PA_DEVERR_TIMEOUT      0x10u /* a bounded wait on a copy expired */
#define PA_DEVERR_APPEND_SLOT  0x20u /* decode_append: slot is not the last position's */
#define PA_DEVERR_QUERY_RANGE  0x40u /* prefill: chunk < 0, > seq_len or > max_query_len */

/* PAGEDATTN_VERSION of the loaded library. */
int pa_version(void);

/* Static, human-readable name of a pa_status. */
const char *pa_status_string(int status);

/*
 * Library plumbing, no passage of the pages behind it: bytes of device
 * workspace pa_decode needs for these sizes (0 when none).  partition_size
 * selects the split-K mode exactly as in pa_decode.  The value depends on the
 * current device's SM count for the split modes.  It takes max_blocks_per_seq
 * (the block-table row length, which bounds every sequence's length) rather
 * than a maximum sequence length, because that is the figure pa_decode itself
 * receives.
 */
size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                int head_dim, int max_blocks_per_seq,
                                int partition_size);

/*
 * Paged decode attention, one query token per sequence.
 *
 * For every sequence s and query head h:
 *     out[s][h] = sum_t softmax_t(scale * q[s][h] . k_t) v_t,   t < seq_lens[s]
 * with k_t, v_t read through block_tables (the block-table figure of the vLLM
 * reading notes: attention addresses non-contiguous KV through the table).
 * The result is the exact softmax attention; scores are never materialised
 * (online softmax with running max and sum, vLLM deep notes, section
 * "核心思想：Tiling + Online Softmax").  A sequence of length 0 yields zeros.
 *
 *   out          [num_seqs][num_heads][head_dim]        dtype, written
 *   q            [num_seqs][num_heads][head_dim]        dtype
 *   k_cache, v_cache  pool, layout above                dtype
 *   block_tables [num_seqs][max_blocks_per_seq] int32;  entries past a
 *                sequence's ceil(len/16) blocks are never read
 *   seq_lens     [num_seqs] int32, 0 <= len <= max_blocks_per_seq * 16
 *   scale        multiplies q.k (typically 1/sqrt(head_dim))
 *
 * Split-K along the sequence (FlashDecoding, ICML tutorial notes, section
 * "内核优化"), chosen by partition_size:
 *   -1  no split: one warp reduces each (sequence, kv head) run whole;
 *    0  balanced split: the grid is sized to the GPU and every warp gets the
 *       same number of 16-token tiles; runs cut by a tile-range boundary are
 *       finished by a log-sum-exp merge.  A batch whose tables are at most
 *       kWholeMaxBlocks = 8 blocks wide and whose (sequence, kv head) runs
 *       number at most four per SM is decoded as with -1 instead (every run
 *       short and on a warp of its own: no merge to wait for);
 *   >0  fixed partitions of partition_size tokens (a multiple of 16); each
 *       partition's partial result is merged with the log-sum-exp rule
 *           M = max_p m_p,  w_p = l_p exp(m_p - M),  o = sum_p w_p o_p / sum_p w_p.
 *       The partials are left at the start of the workspace, fp32, as three
 *       arrays each starting at a 256-byte boundary:
 *           m [num_seqs][num_heads][P_max]  max of the partition's scaled scores
 *           l [num_seqs][num_heads][P_max]  sum_t exp(score_t - m)
 *           o [num_seqs][num_heads][P_max][head_dim]  normalised partial output
 *       P_max = ceil(max_blocks_per_seq * 16 / partition_size); entries of
 *       partitions past a sequence's end, and of sequences that fit one
 *       partition, are not written.  Scratch of the split follows them.
 *
 * A split decode is the decode kernel plus one merge kernel (fixed mode with
 * more than one partition: two).  They are programmatic dependent launches:
 * each may be scheduled while the kernel before it on the stream drains, and
 * touches no global memory until that kernel has completed.
 *
 * workspace: device buffer of at least pa_decode_workspace_size(...) bytes,
 * 256-byte aligned, caller-owned; its contents need no initialisation.  Calls
 * that share a workspace must be ordered on one stream.  The split modes
 * always need one; with no split (-1) a workspace is needed only for batches
 * of more than 2048 sequences, whose per-sequence lengths and tile prefix
 * two small kernels build there first (smaller batches keep them in shared
 * memory).  A batch has no size limit beyond 32-bit tile indices
 * (num_seqs * max_blocks_per_seq * num_kv_heads < 2^31).
 */
int pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, const int32_t *seq_lens,
              int num_seqs, int num_heads, int num_kv_heads, int head_dim,
              int block_size, int max_blocks_per_seq, int num_blocks,
              float scale, int dtype, int partition_size,
              void *workspace, size_t workspace_bytes, void *stream);

/*
 * Chunked-prefill attention over the paged pool: the newest tokens of each
 * sequence (a prompt chunk) attend causally to everything before them and to
 * one another.  Long prompts are cut into chunks that share steps with
 * decodes (vLLM deep notes, section "调度优化：Continuous / Chunked /
 * Disaggregated", part Chunked Prefill; forum summary, section
 * "Sarathi-Serve：Chunked-Prefill技术"); the chunks of a step are packed
 * back to back into one flat batch of rows, as in continuous batching (the
 * same section of the deep notes).
 *
 * Sequence s has seq_lens[s] = L tokens in the pool, its newest
 * c = query_start[s+1] - query_start[s] tokens being the chunk (their K/V
 * are written first, e.g. by pa_reshape_and_cache).  Query row i of the
 * chunk is at position L - c + i and its output is
 *     out[query_start[s] + i, h, :] = sum_{t <= L-c+i} softmax_t(scale q.k_t) v_t
 * with kv head h / (num_heads / num_kv_heads) and k_t, v_t gathered through
 * the block table as in pa_decode.
 *
 *   out, q        [total_q][num_heads][head_dim] dtype, 16-byte aligned;
 *                 total_q = query_start[num_seqs]
 *   query_start   [num_seqs + 1] int32, non-decreasing, query_start[0] = 0
 *   seq_lens      [num_seqs] int32, chunk <= len <= max_blocks_per_seq * 16
 *   max_query_len host copy of the longest chunk: it sizes the grid
 *   scale         > 0
 *   other arguments as in pa_decode.
 * Rows are computed on the fifth-generation tensor cores (S = Q.K^T and
 * O += P.V with fp32 accumulators in tensor memory); P is rounded to dtype
 * before P.V.  A chunk longer than its sequence is skipped and sets
 * PA_DEVERR_QUERY_RANGE; so does one longer than max_query_len, of which
 * only the last max_query_len-ish rows (whole 256-row tiles) are computed.
 * Table entries outside the pool set PA_DEVERR_TABLE_RANGE (block 0 is read
 * instead).
 *
 * workspace (optional, 256-byte aligned, caller-owned, no initialisation
 * needed): at least pa_prefill_workspace_size(...) bytes.  With it a small
 * planning kernel first orders the (sequence, query tile) work: longest
 * first when the batch's K/V fits in L2, so the grid ends on short work (the
 * greedy longest-first schedule); otherwise sequence by sequence, each
 * sequence's kv heads one after the other with all of its query tiles, so
 * that the blocks running together share one head's K/V through L2.
 * Without it (NULL) the work runs in a fixed order.  Results are
 * bit-identical either way.  Calls sharing a workspace must be ordered on
 * one stream.  PA_ERR_WORKSPACE if it is too small or misaligned.
 */
size_t pa_prefill_workspace_size(int num_seqs, int max_query_len, int num_heads,
                                 int num_kv_heads);

int pa_prefill(void *out, const void *q, const void *k_cache, const void *v_cache,
               const int32_t *block_tables, const int32_t *seq_lens, const int32_t *query_start,
               int num_seqs, int max_query_len, int num_heads, int num_kv_heads, int head_dim,
               int block_size, int max_blocks_per_seq, int num_blocks, float scale, int dtype,
               void *workspace, size_t workspace_bytes, void *stream);

/*
 * One decode step with the new tokens appended on the way: the result equals
 *     pa_reshape_and_cache(k_new, v_new, k_cache, v_cache, slot_mapping,
 *                          num_seqs, ...)
 * followed by pa_decode(...), in one launch (plus the merge).  Token s is the
 * newest token of sequence s: slot_mapping[s] must be the slot of position
 * seq_lens[s] - 1 (through block_tables), or negative when sequence s gets
 * no token.  The warp that owns that position's tile takes the row from
 * k_new / v_new directly and writes it to the pool, so no other read of the
 * slot happens in the call.  A slot that is not the last position's is not
 * written and sets PA_DEVERR_APPEND_SLOT.  The block that receives a token
 * must not be read by another sequence in the same call (copy-on-write
 * guarantees this: a shared block is copied before it is written).
 *
 *   k_new, v_new  [num_seqs][num_kv_heads][head_dim]  dtype
 *   slot_mapping  [num_seqs] int64
 * Other arguments as pa_decode; k_cache, v_cache are written.
 */
int pa_decode_append(void *out, const void *q, void *k_cache, void *v_cache,
                     const int32_t *block_tables, const int32_t *seq_lens,
                     const void *k_new, const void *v_new, const int64_t *slot_mapping,
                     int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                     int block_size, int max_blocks_per_seq, int num_blocks,
                     float scale, int dtype, int partition_size,
                     void *workspace, size_t workspace_bytes, void *stream);

/*
 * One decode step of a batch whose sequences come in groups that share a
 * prompt prefix: parallel samples of one prompt keep the prompt's blocks
 * shared by reference (block sharing with copy-on-write, section
 * 系统实现要点 and the page-sharing row of the OS-paging table in the vLLM
 * reading notes).  The result equals pa_decode (or pa_decode_append when
 * k_new, v_new and slot_mapping are given) up to rounding, but each group's
 * shared prefix is read once for the whole group instead of once per
 * sequence: every query column (sample, head) of a group and kv head
 * attends over the prefix together with the others, the prefix's tiles
 * read once through the group's first table (in blocks of up to 64 columns,
 * a long prefix in key chunks); each sequence's own tokens past the prefix
 * are decoded in one decode launch (the tables from the first block past
 * the prefix on, lengths less prefix_len); the partial results
 * of every (sequence, head) are combined with the log-sum-exp rule of the
 * split-K merge.
 *
 *   group_size   sequences [g*group_size, (g+1)*group_size) form group g;
 *                num_seqs must be a multiple of it
 *   prefix_len   tokens of the shared prefix, a multiple of 16, > 0; the
 *                first prefix_len/16 entries of the tables of a group's
 *                sequences must name the same blocks (not checked: the prefix
 *                is read through the group's first table), and every sequence
 *                must be longer than prefix_len when tokens are appended (the
 *                new token must lie past the shared prefix, as copy-on-write
 *                guarantees)
 *   k_new, v_new, slot_mapping  as in pa_decode_append, or all NULL
 *   workspace    at least pa_decode_shared_prefix_workspace_size(...) bytes,
 *                256-byte aligned, caller-owned, no initialisation needed
 * Other arguments as pa_decode.  Launches: the prefix attention (which also
 * writes the suffix lengths), the suffix decode and the final merge (which
 * also folds the pieces of the suffix runs the decode's split cut), all
 * programmatic dependent launches.  A sequence shorter than prefix_len sets
 * PA_DEVERR_SEQLEN_RANGE.
 */
size_t pa_decode_shared_prefix_workspace_size(int num_seqs, int group_size, int prefix_len,
                                              int num_heads, int num_kv_heads, int head_dim,
                                              int max_blocks_per_seq);

int pa_decode_shared_prefix(void *out, const void *q, void *k_cache, void *v_cache,
                            const int32_t *block_tables, const int32_t *seq_lens,
                            const void *k_new, const void *v_new, const int64_t *slot_mapping,
                            int num_seqs, int group_size, int prefix_len, int num_heads,
                            int num_kv_heads, int head_dim, int block_size,
                            int max_blocks_per_seq, int num_blocks, float scale, int dtype,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * pa_decode without a workspace argument, for callers that cannot allocate
 * device memory: an engine that gives (nearly) all free HBM to its KV block
 * pool at start-up and forbids allocations afterwards, a plugin whose host
 * framework hands it only inputs and outputs, or code running where
 * cudaMalloc is not allowed.  The pages describe no such entry point; it has
 * no counterpart there.
 *
 * Same arguments, result and split as pa_decode with partition_size = 0
 * (balanced split).  The split-K scratch is a fixed device array of
 * PA_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads the
 * library holds until the process exits; this call allocates nothing.
 *   - Sizes whose scratch would exceed PA_NOALLOC_SCRATCH_BYTES (see
 *     pa_decode_workspace_size(..., partition_size = 0)) return
 *     PA_ERR_WORKSPACE.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture on the device.
 *   - All calls on a device share the one array and it keeps what the last
 *     call left in it: calls that can overlap on the GPU (different streams,
 *     no ordering between them) race and corrupt each other's results.  Order
 *     them on one stream.
 */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)

int pa_decode_noalloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, const int32_t *seq_lens,
                      int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                      int block_size, int max_blocks_per_seq, int num_blocks,
                      float scale, int dtype, void *stream);

/*
 * Write each new token's K and V into its pool slot: for token i with
 * slot = slot_mapping[i] >= 0, for every kv head h,
 *     k_cache[slot / 16][h][slot % 16][:] = k_new[i][h][:]   (same for V).
 * Blocks are handed out on demand, only when a sequence produces a token
 * that needs a new one, and fill up one token per decode step (forum summary
 * of the notes repository, section 虚拟内存的启示, design point 2; the
 * demand-paging row of the OS-paging table in the vLLM reading notes).
 * Negative slots mark padding tokens and are skipped.  Raw 16-bit copies:
 * bit-exact, NaN payloads preserved.
 *
 *   k_new, v_new  [num_tokens][num_kv_heads][head_dim]  dtype
 *   slot_mapping  [num_tokens] int64
 * Slots >= num_blocks*16 are skipped and set PA_DEVERR_SLOT_RANGE.  Two tokens
 * naming the same slot race (one of them wins).
 */
int pa_reshape_and_cache(const void *k_new, const void *v_new,
                         void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int num_tokens,
                         int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, int dtype, void *stream);

/*
 * Copy-on-write of shared blocks: for every pair i,
 *     k_cache[dst] = k_cache[src], v_cache[dst] = v_cache[src]
 * whole blocks (every kv head and slot), with (src, dst) =
 * block_mapping[i][0], block_mapping[i][1].  Blocks shared by reference
 * count are copied before a sequence writes into them (block sharing for
 * parallel sampling and beam search, the page-sharing row of the OS-paging
 * table and section 系统实现要点 of the vLLM reading notes; reference counts
 * and copy-on-write in the vLLM deep notes, section "PagedAttention：操作系统
 * 启发的设计").
 *
 *   block_mapping [num_pairs][2] int64
 * No dst may appear twice or equal any src (not checked: such pairs race).
 * Pairs naming a block outside the pool are skipped and set
 * PA_DEVERR_BLOCK_RANGE.  Raw 16-bit copies, bit-exact.
 */
int pa_copy_blocks(void *k_cache, void *v_cache, const int64_t *block_mapping,
                   int num_pairs, int num_kv_heads, int head_dim, int block_size,
                   int num_blocks, int dtype, void *stream);

/*
 * Swap blocks between two pools, for preemption: for every pair i,
 *     dst_k[dst] = src_k[src], dst_v[dst] = src_v[src]
 * whole blocks, (src, dst) = block_mapping[i][0], block_mapping[i][1].  One
 * side is the GPU pool, the other a pool of the same layout in page-locked
 * host memory (cudaHostAlloc / cudaHostRegister): blocks of a preempted
 * sequence move to host memory and back instead of being recomputed (the
 * swap row of the OS-paging table and section 系统实现要点 of the vLLM
 * reading notes).  The copy is one kernel reading and writing both pools
 * directly; on GB300 host memory is reached over NVLink-C2C.
 *
 *   src_num_blocks, dst_num_blocks  pool sizes in blocks
 *   block_mapping  [num_pairs][2] int64, device or page-locked host memory
 * Pools must be device memory, managed memory or page-locked host memory;
 * anything else (pageable host memory) returns PA_ERR_INVALID_ARG.  Pairs
 * naming a block outside its pool are skipped and set PA_DEVERR_BLOCK_RANGE.
 * No dst may appear twice (not checked).  Bit-exact.
 */
int pa_swap_blocks(void *dst_k, void *dst_v, const void *src_k, const void *src_v,
                   const int64_t *block_mapping, int num_pairs, int num_kv_heads,
                   int head_dim, int block_size, int src_num_blocks, int dst_num_blocks,
                   int dtype, void *stream);

/*
 * Debug/test export: materialise each sequence's K and V contiguously,
 * read through its block table (the same indirection the decode uses):
 *     k_out[s][h][t][:] = k_cache[block_tables[s][t/16]][h][t%16][:],  t < seq_lens[s]
 *   k_out, v_out  [num_seqs][num_kv_heads][max_blocks_per_seq*16][head_dim];
 *   positions t >= seq_lens[s] are not written.  Bit-exact copies.
 */
int pa_gather_kv(void *k_out, void *v_out, const void *k_cache, const void *v_cache,
                 const int32_t *block_tables, const int32_t *seq_lens,
                 int num_seqs, int num_kv_heads, int head_dim, int block_size,
                 int max_blocks_per_seq, int num_blocks, int dtype, void *stream);

/*
 * Library plumbing, no passage of the pages behind it.  Check the tables a
 * decode would read: counts, into *bad_count (a device uint32 the caller
 * zeroes), the entries block_tables[s][b] with
 * b < ceil(seq_lens[s]/16) outside [0, num_blocks), plus the sequences whose
 * length is outside [0, max_blocks_per_seq*16].
 */
int pa_validate_tables(const int32_t *block_tables, const int32_t *seq_lens,
                       int num_seqs, int max_blocks_per_seq, int num_blocks,
                       int block_size, uint32_t *bad_count, void *stream);

/*
 * Test export for the failure path every copy wait shares: a kernel arms an
 * mbarrier for bytes no copy will deliver and waits with a limit of
 * limit_us microseconds (1..1e6).  The wait must give up, set
 * PA_DEVERR_TIMEOUT and let the kernel finish, leaving the context usable.
 */
int pa_selftest_bounded_wait(int limit_us, void *stream);

/*
 * Library plumbing, no passage of the pages behind it.  Synchronise `stream`,
 * return in *bits the PA_DEVERR_* bits kernels on the current device have
 * recorded since the last clear, and clear them when `clear` is non-zero.
 * Returns PA_ERR_DEVICE when bits is non-zero.  An expired bounded wait is
 * one of those bits (PA_DEVERR_TIMEOUT) rather than a status of its own: the
 * kernel that gave up has long returned when the host asks, and it may have
 * recorded other bits too.
 */
int pa_get_device_error(void *stream, uint32_t *bits, int clear);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
