/*
 * pkv_oracle.c -- the oracle for paged-KV attention.
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the benchmark's
 * CPU-baseline leg are the only users of this file.  The product path (the CUDA
 * library) never loads, links or calls it, and the two share no code, header,
 * table or helper.
 *
 * What it computes is the plain definition, in double precision, with plain loops
 * in the order the definition states them; nothing is blocked, fused or reordered
 * (build without -ffast-math so that no sum is re-associated).
 *
 * Sources (page titles and sections):
 *   [LPNH]   "vLLM推理引擎架构PagedAttention机制与高吞吐推理" (lpnh.cn)
 *            §2.2 BlockManager -- k_cache and v_cache are
 *                 [num_blocks, block_size, num_heads, head_dim];
 *            §2.3 PagedAttention Kernel -- arguments (query [num_tokens, num_heads,
 *                 head_dim], key_cache, value_cache, block_tables [num_seqs,
 *                 max_num_blocks_per_seq], context_lens [num_seqs] = actual length
 *                 of each sequence, block_size); the kernel finds each token's KV
 *                 block through block_tables, scores inside the block and
 *                 accumulates across blocks; output = empty_like(query).
 *   [LESSON] "Servis Motor İçleri: PagedAttention, Sürekli Batching, parçalanmış
 *            Prefill" (aiengineeringfromscratch.com, Phase 17 - 04)
 *            "PagedAttention as a virtual memory system" -- fixed 16-token blocks;
 *                 a block table maps logical token positions to physical block ids;
 *            "Chunked prefill protects the TTFT tail" -- a long prompt runs as
 *                 512-token chunks, each one unit of a batch;
 *            Key Terms -- "Block table", "Chunked prefill".
 *
 * Readings where the pages are silent (each one is listed with its reason in the
 * design notes):
 *   - query head h reads KV head h / (num_heads / num_kv_heads) (consecutive groups);
 *   - slot = physical_block * block_size + offset; a negative slot is a padding
 *     token and is skipped;
 *   - context_lens counts this step's new tokens, which the KV write stores first;
 *   - the q_len rows of a sequence sit at the last q_len positions of its context;
 *     with causal masking row j sees keys 0 .. context_len - q_len + j;
 *   - a sequence with context_len 0 gets an all-zero output;
 *   - an FP8 cache (the pages' headline model runs in FP8: [LESSON], the Llama 3.3
 *     70B FP8 serving numbers) holds OCP e4m3 codes with one scale for K and one for
 *     V: a cached element means code_value * scale; a new element is stored as the
 *     e4m3 code nearest to fp32(x) / scale (one correctly rounded fp32 division),
 *     ties to the even code, magnitudes beyond the largest finite code (448) clamped
 *     to it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#include "pkv_oracle.h"

/* A bf16 value is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * OCP 8-bit floating point, E4M3 variant: sign bit, 4 exponent bits (bias 7), 3
 * mantissa bits.  Exponent field 0 is subnormal (m * 2^-9); exponent field 15 with
 * mantissa 7 is NaN; there are no infinities, so the largest finite value is
 * 1.75 * 2^8 = 448 (code 0x7E).
 */
double oracle_e4m3_decode(uint8_t c)
{
    int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/*
 * The e4m3 code nearest to y: a plain search over the 127 non-negative finite codes
 * (their values increase with the code), ties to the even code; |y| > 448 gives 448;
 * NaN gives 0x7F.  The sign bit is copied (-0.0 -> 0x80).
 */
uint8_t oracle_e4m3_encode(float y)
{
    if (isnan(y)) return 0x7F;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    if (a > 448.0) a = 448.0;
    int best = 0;
    double best_err = a;  /* code 0 has value 0 */
    for (int c = 1; c <= 0x7E; ++c) {
        double err = fabs(oracle_e4m3_decode((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Slot of each new token ([LESSON] "PagedAttention as a virtual memory system":
 * the block table maps a logical token position to a physical block):
 *   slot = block_tables[s][pos / block_size] * block_size + pos % block_size.
 * token_seq[t] < 0 marks a padding token, whose slot is -1.
 */
int oracle_slot_mapping(int64_t *slot_mapping, const int32_t *block_tables,
                        int64_t max_blocks_per_seq, const int32_t *token_seq,
                        const int32_t *token_pos, int64_t num_tokens, int block_size)
{
    for (int64_t t = 0; t < num_tokens; ++t) {
        if (token_seq[t] < 0) {
            slot_mapping[t] = -1;
            continue;
        }
        int64_t pos = token_pos[t];
        if (pos < 0 || pos / block_size >= max_blocks_per_seq) return -1;
        int64_t logical_block = pos / block_size;
        int64_t offset = pos % block_size;
        int64_t physical_block =
            block_tables[(int64_t)token_seq[t] * max_blocks_per_seq + logical_block];
        if (physical_block < 0) return -1;
        slot_mapping[t] = physical_block * block_size + offset;
    }
    return 0;
}

/*
 * KV write ([LPNH] §2.2 cache layout): token t's K row (num_kv_heads x head_dim
 * values) goes to k_cache[slot / block_size][slot % block_size][:][:], same for V.
 * It is a copy of bit patterns.  Returns -1 (having written the valid tokens) if a
 * slot lies outside the pool.
 */
int oracle_reshape_and_cache(uint16_t *k_cache, uint16_t *v_cache, const uint16_t *k,
                             const uint16_t *v, const int64_t *slot_mapping, int64_t num_tokens,
                             int64_t num_blocks, int block_size, int num_kv_heads, int head_dim)
{
    int status = 0;
    int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * block_size) {
            status = -1;
            continue;
        }
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int e = 0; e < head_dim; ++e) {
                int64_t dst = ((block * block_size + offset) * num_kv_heads + h) * head_dim + e;
                int64_t src = t * row + (int64_t)h * head_dim + e;
                k_cache[dst] = k[src];
                v_cache[dst] = v[src];
            }
        }
    }
    return status;
}

/*
 * FP8 KV write: the same placement as above; each element is stored as
 * e4m3(fp32(x) / scale) with x the bf16 value, k_scale for K and v_scale for V.
 */
int oracle_reshape_and_cache_fp8(uint8_t *k_cache, uint8_t *v_cache, const uint16_t *k,
                                 const uint16_t *v, const int64_t *slot_mapping,
                                 int64_t num_tokens, int64_t num_blocks, int block_size,
                                 int num_kv_heads, int head_dim, float k_scale, float v_scale)
{
    if (!(k_scale > 0.0f) || !(v_scale > 0.0f)) return -1;
    int status = 0;
    int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * block_size) {
            status = -1;
            continue;
        }
        const int64_t block = slot / block_size;
        const int64_t offset = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int e = 0; e < head_dim; ++e) {
                int64_t dst = ((block * block_size + offset) * num_kv_heads + h) * head_dim + e;
                int64_t src = t * row + (int64_t)h * head_dim + e;
                float xk = (float)bf16_to_double(k[src]);
                float xv = (float)bf16_to_double(v[src]);
                float yk = xk / k_scale;
                float yv = xv / v_scale;
                k_cache[dst] = oracle_e4m3_encode(yk);
                v_cache[dst] = oracle_e4m3_encode(yv);
            }
        }
    }
    return status;
}

/*
 * Block copy (copy-on-write, [LPNH] §4.3 shared read-only prefix blocks): for each pair
 * (src, dst), every byte of block dst of both caches becomes the byte of block src.
 * Pairs are applied in order.  -1 (having applied the valid pairs) if an id is outside
 * the pool.
 */
int oracle_copy_blocks(uint8_t *k_cache, uint8_t *v_cache, const int32_t *pairs, int64_t num_pairs,
                       int64_t num_blocks, int64_t block_bytes)
{
    int status = 0;
    for (int64_t i = 0; i < num_pairs; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            status = -1;
            continue;
        }
        for (int64_t b = 0; b < block_bytes; ++b) {
            k_cache[dst * block_bytes + b] = k_cache[src * block_bytes + b];
            v_cache[dst * block_bytes + b] = v_cache[src * block_bytes + b];
        }
    }
    return status;
}

/* Check the inputs that decide which memory the attention reads. */
static int check_sequence(const int32_t *block_tables, int64_t max_blocks_per_seq,
                          int64_t num_blocks, int block_size, int64_t s, int64_t ctx,
                          int64_t q_len)
{
    if (ctx < 0 || q_len < 0 || q_len > ctx) return -1;
    if ((ctx + block_size - 1) / block_size > max_blocks_per_seq) return -1;
    for (int64_t i = 0; i < (ctx + block_size - 1) / block_size; ++i) {
        int32_t b = block_tables[s * max_blocks_per_seq + i];
        if (b < 0 || b >= num_blocks) return -1;
    }
    return 0;
}

/*
 * Attention over the paged cache ([LPNH] §2.3), for one (sequence, query head):
 *  1. gather: for every position p < context_len, look up the physical block
 *     block_tables[s][p / block_size] and read row p % block_size of it, building
 *     a contiguous K and V of the sequence for KV head h / group;
 *  2. for each of the sequence's query rows j: logits z_i = scale * <q, K_i> over
 *     the keys it may see, w_i = exp(z_i - max z), out = sum_i w_i V_i / sum_i w_i
 *     (textbook softmax(q K^T scale) V).
 */
static void attend_one(double *out, const uint16_t *q, const void *k_cache,
                       const void *v_cache, int fp8, double k_scale, double v_scale,
                       const int32_t *block_tables,
                       int64_t max_blocks_per_seq, int num_heads, int num_kv_heads, int head_dim,
                       int block_size, double scale, int causal, int64_t s, int h, int64_t ctx,
                       int64_t row0, int64_t q_len, const uint8_t *row_mask)
{
    int group = num_heads / num_kv_heads;
    int hk = h / group;
    double *K = (double *)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1) * head_dim);
    double *V = (double *)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1) * head_dim);
    double *z = (double *)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1));
    double *qd = (double *)malloc(sizeof(double) * (size_t)head_dim);

    /* step 1: gather through the block table */
    for (int64_t p = 0; p < ctx; ++p) {
        int64_t physical = block_tables[s * max_blocks_per_seq + p / block_size];
        int64_t offset = p % block_size;
        for (int e = 0; e < head_dim; ++e) {
            int64_t src = ((physical * block_size + offset) * num_kv_heads + hk) * head_dim + e;
            if (fp8) {
                K[p * head_dim + e] = oracle_e4m3_decode(((const uint8_t *)k_cache)[src]) * k_scale;
                V[p * head_dim + e] = oracle_e4m3_decode(((const uint8_t *)v_cache)[src]) * v_scale;
            } else {
                K[p * head_dim + e] = bf16_to_double(((const uint16_t *)k_cache)[src]);
                V[p * head_dim + e] = bf16_to_double(((const uint16_t *)v_cache)[src]);
            }
        }
    }

    /* step 2: softmax attention per query row */
    for (int64_t j = 0; j < q_len; ++j) {
        int64_t r = row0 + j;
        if (row_mask && !row_mask[r]) continue;
        double *o = out + (r * num_heads + h) * head_dim;
        for (int e = 0; e < head_dim; ++e) qd[e] = bf16_to_double(q[(r * num_heads + h) * head_dim + e]);
        int64_t pos = ctx - q_len + j;
        int64_t n = causal ? pos + 1 : ctx;
        if (n <= 0) {
            for (int e = 0; e < head_dim; ++e) o[e] = 0.0;
            continue;
        }
        double m = -INFINITY;
        for (int64_t i = 0; i < n; ++i) {
            double dot = 0.0;
            for (int e = 0; e < head_dim; ++e) dot += qd[e] * K[i * head_dim + e];
            z[i] = scale * dot;
            if (z[i] > m) m = z[i];
        }
        double denom = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            z[i] = exp(z[i] - m);
            denom += z[i];
        }
        for (int e = 0; e < head_dim; ++e) {
            double acc = 0.0;
            for (int64_t i = 0; i < n; ++i) acc += z[i] * V[i * head_dim + e];
            o[e] = acc / denom;
        }
    }
    free(K);
    free(V);
    free(z);
    free(qd);
}

static int attention(double *out, const uint16_t *q, const void *k_cache, const void *v_cache,
                     int fp8, double k_scale, double v_scale, const int32_t *block_tables,
                     const int32_t *context_lens, const int32_t *query_start_loc,
                     int64_t num_seqs, int64_t max_blocks_per_seq, int num_heads,
                     int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                     double scale, int causal, const uint8_t *row_mask)
{
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return -1;
    if (head_dim <= 0 || block_size <= 0) return -1;
    for (int64_t s = 0; s < num_seqs; ++s) {
        /* A decode row with context_len 0 is an idle batch slot: its output is zero. */
        int64_t q_len = query_start_loc ? query_start_loc[s + 1] - query_start_loc[s]
                                        : (context_lens[s] > 0 ? 1 : 0);
        if (check_sequence(block_tables, max_blocks_per_seq, num_blocks, block_size, s,
                           context_lens[s], q_len) != 0)
            return -1;
    }
    int64_t units = num_seqs * num_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t u = 0; u < units; ++u) {
        int64_t s = u / num_heads;
        int h = (int)(u % num_heads);
        int64_t row0 = query_start_loc ? query_start_loc[s] : s;
        int64_t q_len = query_start_loc ? query_start_loc[s + 1] - query_start_loc[s] : 1;
        attend_one(out, q, k_cache, v_cache, fp8, k_scale, v_scale, block_tables,
                   max_blocks_per_seq, num_heads,
                   num_kv_heads, head_dim, block_size, scale, causal, s, h, context_lens[s], row0,
                   q_len, row_mask);
    }
    return 0;
}

int oracle_paged_attention(double *out, const uint16_t *q, const uint16_t *k_cache,
                           const uint16_t *v_cache, const int32_t *block_tables,
                           const int32_t *context_lens, const int32_t *query_start_loc,
                           int64_t num_seqs, int64_t max_blocks_per_seq, int num_heads,
                           int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                           double scale, int causal, const uint8_t *row_mask)
{
    return attention(out, q, k_cache, v_cache, 0, 1.0, 1.0, block_tables, context_lens,
                     query_start_loc, num_seqs, max_blocks_per_seq, num_heads, num_kv_heads,
                     head_dim, block_size, num_blocks, scale, causal, row_mask);
}

/* The same attention over an FP8 cache: element = e4m3 value of the code * scale. */
int oracle_paged_attention_fp8(double *out, const uint16_t *q, const uint8_t *k_cache,
                               const uint8_t *v_cache, double k_scale, double v_scale,
                               const int32_t *block_tables, const int32_t *context_lens,
                               const int32_t *query_start_loc, int64_t num_seqs,
                               int64_t max_blocks_per_seq, int num_heads, int num_kv_heads,
                               int head_dim, int block_size, int64_t num_blocks, double scale,
                               int causal, const uint8_t *row_mask)
{
    if (!(k_scale > 0.0) || !(v_scale > 0.0)) return -1;
    return attention(out, q, k_cache, v_cache, 1, k_scale, v_scale, block_tables, context_lens,
                     query_start_loc, num_seqs, max_blocks_per_seq, num_heads, num_kv_heads,
                     head_dim, block_size, num_blocks, scale, causal, row_mask);
}
