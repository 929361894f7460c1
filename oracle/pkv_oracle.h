/*
 * pkv_oracle.h -- the oracle's C interface (TEST INFRASTRUCTURE ONLY).
 *
 * Host pointers only.  bf16 data are passed as uint16_t bit patterns; results are
 * double.  Layouts are row-major:
 *   q, out              [total_q_rows, num_heads, head_dim]
 *   k, v (new rows)     [num_tokens, num_kv_heads, head_dim]
 *   k_cache, v_cache    [num_blocks, block_size, num_kv_heads, head_dim]
 *   block_tables        [num_seqs, max_blocks_per_seq]
 *   context_lens        [num_seqs]
 *   query_start_loc     [num_seqs + 1] or NULL (one query row per sequence)
 * Every function returns 0 on success and -1 on an invalid argument.
 */
#ifndef PKV_ORACLE_H
#define PKV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int oracle_num_threads(void);
void oracle_set_num_threads(int n);

int oracle_slot_mapping(int64_t *slot_mapping, const int32_t *block_tables,
                        int64_t max_blocks_per_seq, const int32_t *token_seq,
                        const int32_t *token_pos, int64_t num_tokens, int block_size);

int oracle_reshape_and_cache(uint16_t *k_cache, uint16_t *v_cache, const uint16_t *k,
                             const uint16_t *v, const int64_t *slot_mapping, int64_t num_tokens,
                             int64_t num_blocks, int block_size, int num_kv_heads, int head_dim);

/* row_mask (length total_q_rows) selects the query rows to compute; NULL = all.
 * Rows not selected are left as they were in out. */
int oracle_paged_attention(double *out, const uint16_t *q, const uint16_t *k_cache,
                           const uint16_t *v_cache, const int32_t *block_tables,
                           const int32_t *context_lens, const int32_t *query_start_loc,
                           int64_t num_seqs, int64_t max_blocks_per_seq, int num_heads,
                           int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                           double scale, int causal, const uint8_t *row_mask);

/* Block copy: block dst of both caches (block_bytes bytes each) becomes block src. */
int oracle_copy_blocks(uint8_t *k_cache, uint8_t *v_cache, const int32_t *pairs, int64_t num_pairs,
                       int64_t num_blocks, int64_t block_bytes);

/* FP8 (OCP e4m3) cache: k_cache, v_cache hold one code byte per element.  The codec
 * functions are exported for the tests. */
double oracle_e4m3_decode(uint8_t code);
uint8_t oracle_e4m3_encode(float y);

int oracle_reshape_and_cache_fp8(uint8_t *k_cache, uint8_t *v_cache, const uint16_t *k,
                                 const uint16_t *v, const int64_t *slot_mapping,
                                 int64_t num_tokens, int64_t num_blocks, int block_size,
                                 int num_kv_heads, int head_dim, float k_scale, float v_scale);

int oracle_paged_attention_fp8(double *out, const uint16_t *q, const uint8_t *k_cache,
                               const uint8_t *v_cache, double k_scale, double v_scale,
                               const int32_t *block_tables, const int32_t *context_lens,
                               const int32_t *query_start_loc, int64_t num_seqs,
                               int64_t max_blocks_per_seq, int num_heads, int num_kv_heads,
                               int head_dim, int block_size, int64_t num_blocks, double scale,
                               int causal, const uint8_t *row_mask);

#ifdef __cplusplus
}
#endif

#endif
