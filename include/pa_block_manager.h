/*
 * pa_block_manager.h -- host-side KV block manager (C ABI).
 *
 * Bookkeeping for the block pool the kernels in pagedattn.h read and write,
 * as the vLLM reading notes ("PagedAttention：vLLM 系统论文") describe it in
 * section 系统实现要点 and in the OS-paging table of section 核心思想:
 *   - the pool is allocated once, at start-up; blocks are handed out from a
 *     free list only when a sequence needs one for its next token, and come
 *     back to the free list when no sequence uses them;
 *   - a block can be shared by several sequences (forked samples of one
 *     prompt), tracked by a reference count;
 *   - writing into a shared block first copies it (copy-on-write): the
 *     manager picks a fresh block and reports the (src, dst) pair, which the
 *     caller passes to pa_copy_blocks before the write.
 * The allocation, reference and release events are counted so a caller can
 * observe them (the mini inference engine project of the mlsys-02 course
 * page asks for observable page allocation, references and release).
 *
 * Host memory only; nothing here touches the GPU.  A manager is not
 * thread-safe: calls on one manager must not overlap (a scheduler drives it
 * from one thread).  Sequences are named by caller-chosen 64-bit ids.
 * Every call returns a pa_status from pagedattn.h (PA_OK,
 * PA_ERR_INVALID_ARG, or PA_ERR_OUT_OF_BLOCKS when the free list cannot
 * cover a request; a refused request changes nothing).
 */
#ifndef PA_BLOCK_MANAGER_H
#define PA_BLOCK_MANAGER_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_ERR_OUT_OF_BLOCKS 6   /* the free list cannot cover the request */

typedef struct pa_block_manager pa_block_manager;

typedef struct pa_bm_stats {
    int64_t num_blocks;       /* pool size */
    int64_t free_blocks;      /* blocks on the free list */
    int64_t num_sequences;    /* live sequences */
    int64_t allocations;      /* blocks taken from the free list, ever */
    int64_t releases;         /* blocks returned to the free list, ever */
    int64_t cow_copies;       /* copy-on-write pairs reported, ever */
    int64_t shared_blocks;    /* blocks currently referenced by more than one sequence */
} pa_bm_stats;

/* A manager over a pool of num_blocks blocks of block_size tokens; blocks are
 * handed out lowest id first.  NULL on a bad argument or no memory. */
pa_block_manager *pa_bm_create(int num_blocks, int block_size);
void pa_bm_destroy(pa_block_manager *bm);

/* A new, empty sequence. */
int pa_bm_add_sequence(pa_block_manager *bm, int64_t seq_id);

/* A new sequence `child` that shares every block of `parent` (reference
 * counts go up; no block is copied until one of them writes). */
int pa_bm_fork(pa_block_manager *bm, int64_t parent, int64_t child);

/*
 * Append num_tokens tokens to a sequence.  slots[i] receives the slot
 * (block * block_size + offset) token i is written to -- the slot_mapping of
 * pa_reshape_and_cache.  A new block is taken when a token starts one.  If
 * the first token lands in a shared, partially filled last block, that block
 * is replaced by a fresh copy: the pair (shared block, copy) is written to
 * cow_pairs[0..1] and *num_cow is 1 (else 0); the caller copies it with
 * pa_copy_blocks before writing the tokens.  cow_pairs may be NULL only if
 * the caller knows no copy can happen.
 */
int pa_bm_append(pa_block_manager *bm, int64_t seq_id, int num_tokens, int64_t *slots,
                 int64_t *cow_pairs, int *num_cow);

/* Drop a sequence: its blocks lose one reference and those no longer
 * referenced go back to the free list. */
int pa_bm_free_sequence(pa_block_manager *bm, int64_t seq_id);

/* The sequence's block table (physical block of each logical block) into
 * table[0..max_blocks), padded with -1; *num_blocks and *seq_len receive the
 * counts (either may be NULL).  PA_ERR_INVALID_ARG if the table does not fit. */
int pa_bm_block_table(const pa_block_manager *bm, int64_t seq_id, int32_t *table, int max_blocks,
                      int *num_blocks, int64_t *seq_len);

/* Reference count of a block (0 when free), or -1 for a bad block id. */
int pa_bm_ref_count(const pa_block_manager *bm, int block);

int pa_bm_get_stats(const pa_block_manager *bm, pa_bm_stats *stats);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCK_MANAGER_H */
