/*
 * pda_oracle.h -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow fp64 CPU statement of paged grouped-query decode attention.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library; the CUDA library never includes, links or calls it and
 * this header shares nothing with it.
 *
 * Definition followed (sources cited by page title and section):
 *   - the paged K/V layout [num_blocks, block_size, num_kv_heads, head_dim]
 *     and its element-stride triple (blk, tok, kvh): tiled_attention.rs
 *     (spark_storage), TiledAttention::paged_strides;
 *   - the block list per sequence and the partially filled last block:
 *     tiled_attention.rs, TiledAttention::step_tile (tile_blocks,
 *     tile_block_counts, last_block_valid_slots);
 *   - grouped query heads sharing one KV head, group size
 *     num_q_heads / num_kv_heads: tiled_attention.rs,
 *     TiledAttentionDims::gqa_ratio;
 *   - softmax scale 1/sqrt(head_dim): AstrAI "CUDA Kernels", section
 *     "Python Wrappers" (layout convention);
 *   - the result o / l of the online-softmax state, which is exactly
 *     softmax(scale * q K^T) V: tiled_attention.rs, module comment and
 *     TiledAttention::finalize.
 *
 * Readings taken where the pages are silent: q head h reads KV head
 * h / (num_q_heads / num_kv_heads) (contiguous groups); token t of a sequence
 * lives in block_table[b][t / block_size] at slot t % block_size; a sequence
 * of length 0 yields a zero output row.
 *
 * bf16 values are passed as raw uint16_t bit patterns and widened exactly to
 * double (bits << 16 gives the float32 with the same value).
 */
#ifndef PDA_ORACLE_H
#define PDA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes of the oracle (independent of the CUDA library's codes). */
#define PDO_OK 0
#define PDO_ERR_ARG 1       /* bad sizes, strides or pointers             */
#define PDO_ERR_TABLE 2     /* a block id outside [0, num_blocks)          */
#define PDO_ERR_SEQLEN 3    /* seq_len < 0 or beyond max_blocks*block_size */
#define PDO_ERR_NOMEM 4

/* Exact widening of one bf16 bit pattern to double. */
double pdo_bf16_to_double(uint16_t bits);

/*
 * Attention output for a list of (b, h) pairs.
 *
 *   q           [B, Hq, D] bf16 bits, dense.
 *   k_pool,
 *   v_pool      bf16 bits; row (blk, slot, kvh) starts at element
 *               blk*blk_stride + slot*tok_stride + kvh*kvh_stride and holds
 *               D contiguous elements.
 *   block_table [B, max_blocks] int32 block ids.
 *   seq_lens    [B] int32 token counts.
 *   scale       the softmax scale (callers pass 1/sqrt(D) for the default).
 *   pairs       n_pairs (b, h) pairs as 2*n_pairs int32, or NULL for all
 *               B*Hq pairs in (b, h) row-major order (n_pairs ignored).
 *   n_threads   worker threads (>= 1).
 *   out         [n_pairs][D] doubles (or [B*Hq][D] when pairs is NULL).
 */
int pdo_decode(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
               const int32_t* block_table, const int32_t* seq_lens,
               int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t block_size,
               int64_t num_blocks, int32_t max_blocks,
               int64_t blk_stride, int64_t tok_stride, int64_t kvh_stride,
               double scale, const int32_t* pairs, int64_t n_pairs,
               int32_t n_threads, double* out);

/*
 * Multi-query (causal) decode: q and out are [B, q_len, Hq, D]; seq_lens[b]
 * counts the whole sequence including its last q_len tokens, which are the
 * queries.  Query i of sequence b sits at position seq_lens[b] - q_len + i
 * and attends to tokens 0 .. seq_lens[b] - q_len + i (a causal mask aligned
 * to the end of the sequence; AstrAI "CUDA Kernels", Python Wrappers,
 * is_causal).  A sequence shorter than q_len gives query i the tokens
 * 0 .. max(seq_lens[b] - q_len + i, -1) (none for negative limits: a zero row).
 * out is [B][q_len][Hq][D] doubles.
 */
int pdo_decode_multi(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                     const int32_t* block_table, const int32_t* seq_lens,
                     int32_t B, int32_t q_len, int32_t Hq, int32_t Hkv, int32_t D,
                     int32_t block_size, int64_t num_blocks, int32_t max_blocks,
                     int64_t blk_stride, int64_t tok_stride, int64_t kvh_stride,
                     double scale, int32_t n_threads, double* out);

/*
 * The block-table gather on its own: copies the K and V rows of sequence b,
 * KV head kvh, tokens 0..seq_lens[b]-1 in order, into k_rows / v_rows
 * ([seq_lens[b]][D] bf16 bits each).
 */
int pdo_gather(const uint16_t* k_pool, const uint16_t* v_pool,
               const int32_t* block_table, const int32_t* seq_lens,
               int32_t B, int32_t Hkv, int32_t D, int32_t block_size,
               int64_t num_blocks, int32_t max_blocks,
               int64_t blk_stride, int64_t tok_stride, int64_t kvh_stride,
               int32_t b, int32_t kvh, uint16_t* k_rows, uint16_t* v_rows);

#ifdef __cplusplus
}
#endif

#endif /* PDA_ORACLE_H */
