/*
 * oracle.c -- plain, slow, fp64 CPU reference for paged decode attention,
 * chunked-prefill attention over the same pool, and the KV-pool maintenance
 * operations (slot scatter, block copy, swap between pools).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this code; only the
 * tests, the smoke check and the benchmark's CPU-baseline leg load it.  It
 * shares no code, header or table with the CUDA path.
 *
 * What it computes (the pages' statement of the problem):
 *   - K/V of a sequence live in fixed 16-token blocks of a preallocated pool;
 *     token t of sequence s sits in physical block block_tables[s][t / 16] at
 *     offset t % 16, and attention reads K/V indirectly through that table
 *     ("PagedAttention: Efficient Memory Management for LLM Serving" reading
 *     notes, section 核心思想, block-table figure and the OS-paging table).
 *   - Paging only changes addressing, so the decode result is plain
 *     single-query softmax attention over the sequence's tokens.  Exact
 *     attention is what the FlashAttention family also returns (vLLM deep
 *     notes, section "FlashAttention: IO-Aware 精确注意力").
 *   - Grouped-query attention: several query heads share one K/V head (ICML
 *     tutorial notes, section "Attention 简化与 KV Cache 优化").  Query head h
 *     reads kv head h / G, G = num_heads / num_kv_heads (contiguous groups).
 *   - Split-K over the sequence (FlashDecoding, ICML tutorial notes, section
 *     "内核优化"): a partition's partial result and the log-sum-exp merge of
 *     partials, each written as its plain definition.
 *   - Chunked prefill (vLLM deep notes, section "调度优化：Continuous /
 *     Chunked / Disaggregated"): the newest c tokens of a sequence of length
 *     L are a chunk whose K/V are already in the pool; chunk row i sits at
 *     position L - c + i and attends to positions 0 .. L - c + i, the same
 *     single-row attention as a decode over that prefix.
 *
 * Layouts (shared with the library by convention, not by code):
 *   q        [num_seqs][num_heads][D]                 fp16/bf16 bits
 *            (prefill: [total_rows][num_heads][D], chunks back to back,
 *            query_start [num_seqs + 1] int32)
 *   k/v pool [num_blocks][num_kv_heads][16][D]         fp16/bf16 bits
 *   block_tables [num_seqs][max_blocks_per_seq] int32, seq_lens [num_seqs] int32
 *
 * All arithmetic is double precision, every input is decoded from its 16-bit
 * pattern exactly, and nothing is blocked, fused or reordered beyond the
 * definition.  The functions are single-threaded; callers may run disjoint
 * ranges of sequences on separate threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(f + 1024), e - 25);    /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -mag : mag;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double decode_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

static double decode(uint16_t bits, int dtype)
{
    return dtype == ORACLE_BF16 ? decode_bf16(bits) : decode_f16(bits);
}

/* Decode n 16-bit patterns to double (exposed so tests can pin the decoders). */
void oracle_decode_bits(double *out, const uint16_t *bits, long n, int dtype)
{
    for (long i = 0; i < n; ++i)
        out[i] = decode(bits[i], dtype);
}

/* Address of element d of token t (of kv head kvh) for sequence s, found
 * through the block table. */
static long pool_index(const int32_t *block_tables, int max_blocks_per_seq,
                       int num_kv_heads, int block_size, int head_dim,
                       int s, int kvh, int t, int d)
{
    long phys = block_tables[(long)s * max_blocks_per_seq + t / block_size];
    int off = t % block_size;
    return ((phys * num_kv_heads + kvh) * block_size + off) * (long)head_dim + d;
}

/*
 * Attention of query head h of sequence s over its tokens [t0, t1).
 *   x_t = scale * sum_d q_d k_{t,d}
 *   m   = max_t x_t
 *   l   = sum_t exp(x_t - m)
 *   o   = sum_t exp(x_t - m) v_t / l
 * With [t0, t1) = [0, seq_len) `o` is the decode output; with a partition it
 * is that partition's partial result (m, l, o).  An empty range gives
 * m = -inf, l = 0, o = 0.  The score vector is kept whole, as in dense
 * softmax: no running max, no tiling.
 */
static void attend_row(double *o, double *m_out, double *l_out, const uint16_t *qh,
                       const uint16_t *k_cache, const uint16_t *v_cache,
                       const int32_t *block_tables, int max_blocks_per_seq,
                       int num_heads, int num_kv_heads, int head_dim, int block_size,
                       double scale, int dtype, int s, int h, int t0, int t1);

void oracle_attend(double *o, double *m_out, double *l_out,
                   const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                   const int32_t *block_tables, int max_blocks_per_seq,
                   int num_heads, int num_kv_heads, int head_dim, int block_size,
                   double scale, int dtype, int s, int h, int t0, int t1)
{
    attend_row(o, m_out, l_out, q + ((long)s * num_heads + h) * head_dim, k_cache, v_cache,
               block_tables, max_blocks_per_seq, num_heads, num_kv_heads, head_dim, block_size,
               scale, dtype, s, h, t0, t1);
}

/* The attention of one query row qh (query head h of sequence s) over the
 * sequence's tokens [t0, t1); see oracle_attend. */
static void attend_row(double *o, double *m_out, double *l_out, const uint16_t *qh,
                       const uint16_t *k_cache, const uint16_t *v_cache,
                       const int32_t *block_tables, int max_blocks_per_seq,
                       int num_heads, int num_kv_heads, int head_dim, int block_size,
                       double scale, int dtype, int s, int h, int t0, int t1)
{
    int D = head_dim;
    int G = num_heads / num_kv_heads;
    int kvh = h / G;
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    if (t1 <= t0) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return;
    }
    int n = t1 - t0;
    double *x = (double *)malloc(sizeof(double) * (size_t)n);
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    for (int d = 0; d < D; ++d)
        qd[d] = decode(qh[d], dtype);
    /* scores */
    for (int i = 0; i < n; ++i) {
        int t = t0 + i;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) {
            long at = pool_index(block_tables, max_blocks_per_seq, num_kv_heads,
                                 block_size, D, s, kvh, t, d);
            acc += qd[d] * decode(k_cache[at], dtype);
        }
        x[i] = scale * acc;
    }
    /* max-subtracted softmax weights */
    double m = x[0];
    for (int i = 1; i < n; ++i)
        if (x[i] > m)
            m = x[i];
    double l = 0.0;
    for (int i = 0; i < n; ++i) {
        x[i] = exp(x[i] - m);
        l += x[i];
    }
    /* weighted sum of values */
    for (int i = 0; i < n; ++i) {
        int t = t0 + i;
        for (int d = 0; d < D; ++d) {
            long at = pool_index(block_tables, max_blocks_per_seq, num_kv_heads,
                                 block_size, D, s, kvh, t, d);
            o[d] += x[i] * decode(v_cache[at], dtype);
        }
    }
    for (int d = 0; d < D; ++d)
        o[d] /= l;
    *m_out = m;
    *l_out = l;
    free(x);
    free(qd);
}

/*
 * Decode output for sequences [seq_begin, seq_end), every query head:
 * out[s][h][d] (double).  A sequence of length 0 has no tokens to attend to;
 * its output is defined as zeros.
 */
void oracle_decode(double *out, const uint16_t *q, const uint16_t *k_cache,
                   const uint16_t *v_cache, const int32_t *block_tables,
                   const int32_t *seq_lens, int num_heads, int num_kv_heads,
                   int head_dim, int block_size, int max_blocks_per_seq,
                   double scale, int dtype, int seq_begin, int seq_end)
{
    for (int s = seq_begin; s < seq_end; ++s) {
        for (int h = 0; h < num_heads; ++h) {
            double m, l;
            double *o = out + ((long)s * num_heads + h) * head_dim;
            oracle_attend(o, &m, &l, q, k_cache, v_cache, block_tables,
                          max_blocks_per_seq, num_heads, num_kv_heads, head_dim,
                          block_size, scale, dtype, s, h, 0, seq_lens[s]);
        }
    }
}

/*
 * Split-K partials of sequences [seq_begin, seq_end): partition p covers
 * tokens [p*P, min((p+1)*P, L)).  Layout m/l [num_seqs][num_heads][P_max],
 * o [num_seqs][num_heads][P_max][D].  Partitions past the sequence's end are
 * left untouched.
 */
void oracle_partials(double *m_out, double *l_out, double *o_out,
                     const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                     const int32_t *block_tables, const int32_t *seq_lens,
                     int num_heads, int num_kv_heads, int head_dim, int block_size,
                     int max_blocks_per_seq, double scale, int dtype,
                     int partition_size, int max_partitions,
                     int seq_begin, int seq_end)
{
    for (int s = seq_begin; s < seq_end; ++s) {
        int L = seq_lens[s];
        int np = (L + partition_size - 1) / partition_size;
        for (int h = 0; h < num_heads; ++h) {
            for (int p = 0; p < np && p < max_partitions; ++p) {
                long row = ((long)s * num_heads + h) * max_partitions + p;
                int t0 = p * partition_size;
                int t1 = t0 + partition_size < L ? t0 + partition_size : L;
                oracle_attend(o_out + row * head_dim, m_out + row, l_out + row,
                              q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                              num_heads, num_kv_heads, head_dim, block_size,
                              scale, dtype, s, h, t0, t1);
            }
        }
    }
}

/*
 * Log-sum-exp merge of n partials (m_p, l_p, o_p) of one head:
 *   M   = max_p m_p
 *   w_p = l_p * exp(m_p - M)
 *   o   = sum_p w_p o_p / sum_p w_p
 * Partials with l_p = 0 (empty partitions) carry no weight.
 */
void oracle_lse_merge(double *o, const double *m, const double *l,
                      const double *op, int n, int head_dim)
{
    double M = -INFINITY;
    for (int p = 0; p < n; ++p)
        if (l[p] > 0.0 && m[p] > M)
            M = m[p];
    double W = 0.0;
    for (int d = 0; d < head_dim; ++d)
        o[d] = 0.0;
    for (int p = 0; p < n; ++p) {
        if (!(l[p] > 0.0))
            continue;
        double w = l[p] * exp(m[p] - M);
        W += w;
        for (int d = 0; d < head_dim; ++d)
            o[d] += w * op[(long)p * head_dim + d];
    }
    for (int d = 0; d < head_dim; ++d)
        o[d] = W > 0.0 ? o[d] / W : 0.0;
}

/*
 * Contiguous K and V of sequence s, all kv heads, gathered through the block
 * table: out[kvh][t][d] for t < seq_len (raw 16-bit copies).
 */
void oracle_gather_kv(uint16_t *k_out, uint16_t *v_out, const uint16_t *k_cache,
                      const uint16_t *v_cache, const int32_t *block_tables,
                      int max_blocks_per_seq, int num_kv_heads, int head_dim,
                      int block_size, int s, int seq_len)
{
    for (int kvh = 0; kvh < num_kv_heads; ++kvh)
        for (int t = 0; t < seq_len; ++t)
            for (int d = 0; d < head_dim; ++d) {
                long at = pool_index(block_tables, max_blocks_per_seq, num_kv_heads,
                                     block_size, head_dim, s, kvh, t, d);
                long to = ((long)kvh * seq_len + t) * head_dim + d;
                k_out[to] = k_cache[at];
                v_out[to] = v_cache[at];
            }
}

/*
 * Write each new token's K and V (all kv heads) into pool slot
 * slot_mapping[i] = block * block_size + offset.  Negative slots mark padding
 * tokens and are skipped; slots past the pool are skipped too and counted in
 * the return value.
 */
long oracle_reshape_and_cache(uint16_t *k_cache, uint16_t *v_cache,
                              const uint16_t *k_new, const uint16_t *v_new,
                              const int64_t *slot_mapping, int num_tokens,
                              int num_kv_heads, int head_dim, int block_size,
                              long num_blocks)
{
    long bad = 0;
    for (int i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        if (slot >= num_blocks * block_size) {
            ++bad;
            continue;
        }
        long blk = (long)(slot / block_size);
        int off = (int)(slot % block_size);
        for (int kvh = 0; kvh < num_kv_heads; ++kvh)
            for (int d = 0; d < head_dim; ++d) {
                long to = ((blk * num_kv_heads + kvh) * block_size + off) * (long)head_dim + d;
                long from = ((long)i * num_kv_heads + kvh) * head_dim + d;
                k_cache[to] = k_new[from];
                v_cache[to] = v_new[from];
            }
    }
    return bad;
}

/*
 * Copy-on-write: for each (src, dst) pair copy the whole block (every kv head,
 * every slot) of K and of V.  Pairs naming a block outside the pool are
 * skipped and counted in the return value.
 */
long oracle_copy_blocks(uint16_t *k_cache, uint16_t *v_cache,
                        const int64_t *block_mapping, int num_pairs,
                        int num_kv_heads, int head_dim, int block_size, long num_blocks)
{
    long bad = 0;
    long per_block = (long)num_kv_heads * block_size * head_dim;
    for (int i = 0; i < num_pairs; ++i) {
        int64_t src = block_mapping[2 * i];
        int64_t dst = block_mapping[2 * i + 1];
        if (src < 0 || dst < 0 || src >= num_blocks || dst >= num_blocks) {
            ++bad;
            continue;
        }
        for (long e = 0; e < per_block; ++e) {
            k_cache[dst * per_block + e] = k_cache[src * per_block + e];
            v_cache[dst * per_block + e] = v_cache[src * per_block + e];
        }
    }
    return bad;
}

/*
 * Swap: for each (src, dst) pair copy block src of the source pools into
 * block dst of the destination pools (every kv head and slot, K and V).  One
 * pool side is GPU memory, the other host memory: preempted sequences' blocks
 * move to host memory and back (the swap row of the OS-paging table and
 * section 系统实现要点 of the vLLM reading notes).  Pairs naming a block
 * outside its pool are skipped and counted in the return value.
 */
long oracle_swap_blocks(uint16_t *dst_k, uint16_t *dst_v, const uint16_t *src_k,
                        const uint16_t *src_v, const int64_t *block_mapping, int num_pairs,
                        int num_kv_heads, int head_dim, int block_size, long src_blocks,
                        long dst_blocks)
{
    long bad = 0;
    long per_block = (long)num_kv_heads * block_size * head_dim;
    for (int i = 0; i < num_pairs; ++i) {
        int64_t src = block_mapping[2 * i];
        int64_t dst = block_mapping[2 * i + 1];
        if (src < 0 || dst < 0 || src >= src_blocks || dst >= dst_blocks) {
            ++bad;
            continue;
        }
        for (long e = 0; e < per_block; ++e) {
            dst_k[dst * per_block + e] = src_k[src * per_block + e];
            dst_v[dst * per_block + e] = src_v[src * per_block + e];
        }
    }
    return bad;
}

/*
 * Paged prefill of a chunk of new tokens per sequence (chunked prefill, the
 * Sarathi-Serve scheme in the notes: a long prompt is processed in chunks,
 * interleaved with decode steps).  The chunk of sequence s is rows
 * query_start[s] .. query_start[s+1] of q ([total][num_heads][D]); they are
 * the last positions of the sequence, whose length seq_lens[s] includes the
 * chunk, and their K/V are already in the pool.  Row i of the chunk sits at
 * position p = seq_lens[s] - chunk + i and attends causally to tokens 0..p.
 * out[row][h][d] (double), for sequences [seq_begin, seq_end).
 */
void oracle_prefill(double *out, const uint16_t *q, const uint16_t *k_cache,
                    const uint16_t *v_cache, const int32_t *block_tables,
                    const int32_t *seq_lens, const int32_t *query_start, int num_heads,
                    int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                    double scale, int dtype, int seq_begin, int seq_end)
{
    for (int s = seq_begin; s < seq_end; ++s) {
        int chunk = query_start[s + 1] - query_start[s];
        for (int i = 0; i < chunk; ++i) {
            long row = query_start[s] + i;
            int p = seq_lens[s] - chunk + i;
            for (int h = 0; h < num_heads; ++h) {
                double m, l;
                attend_row(out + (row * num_heads + h) * head_dim, &m, &l,
                           q + (row * num_heads + h) * head_dim, k_cache, v_cache,
                           block_tables, max_blocks_per_seq, num_heads, num_kv_heads,
                           head_dim, block_size, scale, dtype, s, h, 0, p + 1);
            }
        }
    }
}
