/*
 * pagedkv.h -- C ABI of libpagedkv.so: attention over a block-paged KV cache on
 * NVIDIA GB300 (sm_103a).
 *
 * The operations follow two descriptions of the method:
 *   [LPNH]   "vLLM推理引擎架构PagedAttention机制与高吞吐推理" (lpnh.cn):
 *            §2.2 BlockManager (allocate / free over a pool of fixed-size blocks;
 *            k_cache and v_cache shaped [num_blocks, block_size, num_heads,
 *            head_dim]); §2.3 PagedAttention Kernel (query, key_cache,
 *            value_cache, block_tables, context_lens, block_size; look up each
 *            token's block through block_tables, score inside the block,
 *            accumulate across blocks; output = empty_like(query)); §4.1 block
 *            size (default 16).
 *   [LESSON] "Servis Motor İçleri: PagedAttention, Sürekli Batching, parçalanmış
 *            Prefill" (aiengineeringfromscratch.com, Phase 17 - 04):
 *            "PagedAttention as a virtual memory system" (a block table maps
 *            logical token positions to physical block ids; a sequence gains one
 *            block when it grows past the ones it holds); "Chunked prefill
 *            protects the TTFT tail" (512-token prompt chunks scheduled next to
 *            single-token decodes); "What the scheduler looks like" (one fused GPU
 *            call per iteration).
 *
 * Conventions for every call below
 *   - Device pointers are CUDA device memory owned by the caller; the library
 *     never allocates, frees or keeps them.  Host pointers are named host_*.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Kernels are
 *     launched asynchronously on it; nothing is copied back to the host, so a
 *     call returns before the GPU has finished.
 *   - Layouts are row-major and dense:
 *       q, out                 [tokens, num_heads, head_dim]          bf16
 *       k, v (new rows)        [num_tokens, num_kv_heads, head_dim]   bf16
 *       k_cache, v_cache       [num_blocks, block_size, num_kv_heads, head_dim] bf16
 *       block_tables           [num_seqs, max_blocks_per_seq]         int32
 *       context_lens           [num_seqs]                             int32
 *       query_start_loc        [num_seqs + 1], query_start_loc[0] = 0 int32
 *       slot_mapping           [num_tokens]                           int64
 *   - Query head h reads KV head h / (num_heads / num_kv_heads).
 *   - context_lens[s] counts every token of sequence s in the cache, this step's
 *     new tokens included (write them with pkv_reshape_and_cache first).  A
 *     sequence's q_len query rows are its last q_len positions.
 *   - Accumulation is fp32; outputs are rounded to bf16 (round to nearest even).
 *   - Return value: PKV_OK or a negative PKV_ERR_* code, for argument errors the
 *     host can see.  Errors in device data (a block id outside the pool, a slot
 *     outside the pool, a context longer than its block-table row, q_len larger
 *     than context_len) cannot be seen by the host: the kernels skip the bad
 *     item, never read or write outside the caller's buffers, and record a flag
 *     in a device error word that pkv_get_device_error returns.
 *   - Per-device state: on its first call on a device (with that device current) the
 *     library looks up facts it then keeps for the life of the process -- the SM count,
 *     the shared-memory limit, and the device addresses of its own device variables
 *     (the error word, the static scratch array).  These lookups assume the device's
 *     primary context is never reset or destroyed while the library is loaded
 *     (cudaDeviceReset, or a context torn down and created again, would leave the kept
 *     addresses stale).  Make the first call on a device before any stream capture.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes --------------------------------------------------------- */
#define PKV_OK                       0
#define PKV_ERR_INVALID_ARG         -1  /* null pointer, negative or inconsistent size */
#define PKV_ERR_UNSUPPORTED         -2  /* valid but not built: see each call */
#define PKV_ERR_WORKSPACE_TOO_SMALL -3  /* workspace_bytes < pkv_workspace_size(...) */
#define PKV_ERR_CUDA                -4  /* a CUDA runtime call or launch failed */
#define PKV_ERR_OOM                 -5  /* block manager: not enough free blocks */
#define PKV_ERR_DEVICE_DATA         -6  /* returned by pkv_get_device_error */
#define PKV_ERR_STATIC_SCRATCH_LIMIT -7 /* sizes need more than PKV_STATIC_SCRATCH_BYTES */

/* ---- flags in the device error word (pkv_get_device_error) ---------------- */
#define PKV_DEVERR_SLOT         0x1   /* slot_mapping entry >= num_blocks * block_size */
#define PKV_DEVERR_BLOCK_ID     0x2   /* block_tables entry outside [0, num_blocks) */
#define PKV_DEVERR_CONTEXT_LEN  0x4   /* context_len < 0 or > max_blocks_per_seq * block_size */
#define PKV_DEVERR_QUERY_LEN    0x8   /* q_len < 0 or q_len > context_len */
#define PKV_DEVERR_TIMEOUT      0x10  /* a pipeline wait gave up (internal fault) */

/* ---- dtypes --------------------------------------------------------------- */
#define PKV_DTYPE_BF16 0
/* An FP8 cache: one OCP e4m3 code byte per element (the pages' headline model,
 * Llama 3.3 70B, is served in FP8: [LESSON] "Numbers you should remember").  Used
 * through the *_fp8 calls below, which take the per-tensor scales. */
#define PKV_DTYPE_FP8_E4M3 1

/* ---- ops for pkv_workspace_size ------------------------------------------- */
#define PKV_OP_DECODE 0
#define PKV_OP_VARLEN 1

/*
 * KV write ("reshape_and_cache").  [LPNH] §2.2 pool layout; [LESSON] "PagedAttention
 * as a virtual memory system" (a token's K/V row lives in one slot of a block).
 * For each token t with slot = slot_mapping[t] >= 0:
 *     k_cache[slot / block_size][slot % block_size][:][:] = k[t][:][:]   (same for v)
 * A negative slot marks a padding token and is skipped.  The copy is bit-exact.
 * Slots >= num_blocks * block_size are skipped and flagged PKV_DEVERR_SLOT.
 * Two tokens with the same slot race (the result is one of them).
 * Supported: dtype PKV_DTYPE_BF16, num_kv_heads * head_dim a multiple of 8.
 */
int pkv_reshape_and_cache(void *k_cache, void *v_cache, const void *k, const void *v,
                          const int64_t *slot_mapping, int64_t num_tokens, int64_t num_blocks,
                          int block_size, int num_kv_heads, int head_dim, int dtype,
                          void *stream);

/*
 * Decode attention: one query row per sequence.  [LPNH] §2.3.
 * For sequence s and query head h (KV head hk = h / (num_heads / num_kv_heads)):
 *     out[s][h] = softmax(scale * q[s][h] . K_s^T) V_s
 * where K_s, V_s are rows 0 .. context_lens[s]-1 of the sequence, row p stored in
 * block block_tables[s][p / block_size], slot p % block_size.  context_lens[s] = 0
 * gives a zero row.  Long contexts are split across thread blocks and the parts
 * merged with their log-sum-exp weights; `workspace` (device, >=
 * pkv_workspace_size(PKV_OP_DECODE, ...) bytes, 256-byte aligned, contents
 * irrelevant on entry) holds the parts.  Calls that share a workspace must be
 * ordered on one stream.
 * Supported: dtype bf16, block_size 8, 16, 32 or 64, head_dim 64 or 128, num_heads a
 * multiple of num_kv_heads, group = num_heads / num_kv_heads <= 64, num_seqs <= 4096.
 */
int pkv_paged_attention_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *block_tables, const int32_t *context_lens,
                               int num_seqs, int max_blocks_per_seq, int num_heads,
                               int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                               float scale, int dtype, void *workspace, size_t workspace_bytes,
                               void *stream);

/*
 * FP8 KV cache (e4m3 codes, one scale for K and one for V).  The pages state the
 * cache layout and name FP8 serving but not the element encoding; the reading
 * here: a cached code c means e4m3_value(c) * scale, where e4m3 is the OCP 8-bit
 * floating-point format E4M3 (bias 7, 3 mantissa bits, subnormals, largest finite
 * 448, NaN = S.1111.111, no infinities).
 *
 * pkv_reshape_and_cache_fp8: the same placement as pkv_reshape_and_cache; k and v
 * are bf16 rows, k_cache and v_cache uint8 [num_blocks, block_size, num_kv_heads,
 * head_dim].  Element x of a K row is stored as the e4m3 code nearest to
 * fp32(x) / k_scale (one correctly rounded fp32 division), ties to the even code,
 * magnitudes beyond 448 stored as +-448; likewise v with v_scale.  Bit-exact.
 * Scales must be finite and > 0 (else PKV_ERR_INVALID_ARG).
 * Supported: num_kv_heads * head_dim a multiple of 16.
 */
int pkv_reshape_and_cache_fp8(void *k_cache, void *v_cache, const void *k, const void *v,
                              const int64_t *slot_mapping, int64_t num_tokens,
                              int64_t num_blocks, int block_size, int num_kv_heads,
                              int head_dim, float k_scale, float v_scale, void *stream);

/*
 * pkv_paged_attention_decode_fp8: pkv_paged_attention_decode over an FP8 cache,
 * with every cached K element read as e4m3_value * k_scale and every V element as
 * e4m3_value * v_scale.  q and out stay bf16.  On the tensor cores the products
 * run in fp16 with fp32 accumulation: the e4m3 codes widen to fp16 exactly, q is
 * rounded to fp16 (exact for bf16 values of magnitude in [2^-14, 65504]), the
 * softmax weights are rounded to fp16.  Workspace as for the bf16 call
 * (pkv_workspace_size(PKV_OP_DECODE, ...)).
 * Supported: block_size 8, 16, 32 or 64, head_dim 128, the bf16 call's head counts.
 */
int pkv_paged_attention_decode_fp8(void *out, const void *q, const void *k_cache,
                                   const void *v_cache, const int32_t *block_tables,
                                   const int32_t *context_lens, int num_seqs,
                                   int max_blocks_per_seq, int num_heads, int num_kv_heads,
                                   int head_dim, int block_size, int64_t num_blocks, float scale,
                                   float k_scale, float v_scale, void *workspace,
                                   size_t workspace_bytes, void *stream);

/*
 * Decode step with its KV write fused into the attention launch.  For every sequence s
 * with context_lens[s] >= 1, the rows k_new[s] and v_new[s] (k_new, v_new [num_seqs,
 * num_kv_heads, head_dim] bf16, device) are stored at position p = context_lens[s] - 1
 * -- block block_tables[s][p / block_size], offset p % block_size -- and then
 * out[s] = decode attention over positions 0 .. p, exactly as pkv_slot_mapping of those
 * positions + pkv_reshape_and_cache (resp. pkv_reshape_and_cache_fp8) +
 * pkv_paged_attention_decode (resp. _fp8) would give, in one launch (plus the merge).
 * The thread block that reads a sequence's last 16 positions writes its new rows first.
 * Arguments, support and errors as for pkv_paged_attention_decode (dtype must be
 * PKV_DTYPE_BF16) and pkv_paged_attention_decode_fp8; k_new and v_new 16-byte aligned.
 * A block id outside the pool at position p skips that write (PKV_DEVERR_BLOCK_ID).
 */
int pkv_paged_attention_decode_kvwrite(void *out, const void *q, const void *k_new, const void *v_new,
                                       void *k_cache, void *v_cache, const int32_t *block_tables,
                                       const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                                       int num_heads, int num_kv_heads, int head_dim, int block_size,
                                       int64_t num_blocks, float scale, int dtype, void *workspace,
                                       size_t workspace_bytes, void *stream);
int pkv_paged_attention_decode_kvwrite_fp8(void *out, const void *q, const void *k_new,
                                           const void *v_new, void *k_cache, void *v_cache,
                                           const int32_t *block_tables, const int32_t *context_lens,
                                           int num_seqs, int max_blocks_per_seq, int num_heads,
                                           int num_kv_heads, int head_dim, int block_size,
                                           int64_t num_blocks, float scale, float k_scale,
                                           float v_scale, void *workspace, size_t workspace_bytes,
                                           void *stream);

/*
 * Block copy (the device half of copy-on-write, [LPNH] §4.3): for each i < num_pairs,
 * with (src, dst) = (block_pairs[2i], block_pairs[2i+1]) (device int32),
 *     k_cache[dst] = k_cache[src]  and  v_cache[dst] = v_cache[src]   (whole blocks)
 * of a pool laid out as [num_blocks, block_size, num_kv_heads, head_dim] with elements
 * of `dtype` (PKV_DTYPE_BF16 or PKV_DTYPE_FP8_E4M3).  Bit-exact.  A dst must not appear
 * as another pair's src or dst in the same call (the copies run in parallel).  Ids outside
 * the pool are skipped and flagged PKV_DEVERR_BLOCK_ID.
 */
int pkv_copy_blocks(void *k_cache, void *v_cache, const int32_t *block_pairs, int64_t num_pairs,
                    int64_t num_blocks, int block_size, int num_kv_heads, int head_dim, int dtype,
                    void *stream);

/*
 * Varlen attention over a ragged batch in one call ([LESSON] "Chunked prefill
 * protects the TTFT tail", "What the scheduler looks like": prefill chunks and
 * single-token decodes in one fused GPU call).  Sequence s owns query rows
 * query_start_loc[s] .. query_start_loc[s+1]-1, at positions
 * context_lens[s] - q_len .. context_lens[s] - 1.  With causal != 0, row j of a
 * sequence sees keys 0 .. context_lens[s] - q_len + j; otherwise all
 * context_lens[s] keys.  q_len = 1 rows take the decode path; longer ones the
 * chunked-prefill path.  total_q_tokens = query_start_loc[num_seqs] and max_q_len
 * bounds every q_len (both as the caller knows them on the host).
 * Supported: as for decode, plus total_q_tokens <= 2^31 - 1; rows with q_len >= 2
 * need block_size 16 and group = num_heads / num_kv_heads <= 8 (PKV_ERR_UNSUPPORTED
 * otherwise).
 */
int pkv_paged_attention_varlen(void *out, const void *q, const int32_t *query_start_loc,
                               const void *k_cache, const void *v_cache,
                               const int32_t *block_tables, const int32_t *context_lens,
                               int num_seqs, int total_q_tokens, int max_q_len,
                               int max_blocks_per_seq, int num_heads, int num_kv_heads,
                               int head_dim, int block_size, int64_t num_blocks, float scale,
                               int causal, int dtype, void *workspace, size_t workspace_bytes,
                               void *stream);

/*
 * pkv_paged_attention_varlen_fp8: pkv_paged_attention_varlen over an FP8 cache (the
 * encoding of pkv_reshape_and_cache_fp8): every cached K element reads as
 * e4m3_value * k_scale and every V element as e4m3_value * v_scale; q and out stay
 * bf16.  Single-token rows take the FP8 decode path (pkv_paged_attention_decode_fp8);
 * multi-token rows run on the tensor cores in fp16 with fp32 accumulation: the codes
 * widen to fp16 exactly, q is rounded to fp16, the softmax weights are rounded to fp16.
 * Pool rows at or past a sequence's context are never read as values (they may hold
 * any code, NaN included).  Workspace: pkv_workspace_size(PKV_OP_VARLEN, ...).
 * Scales must be finite and > 0 (else PKV_ERR_INVALID_ARG).
 * Supported: head_dim 128, block_size 16 when any row has q_len >= 2 (8, 16, 32 or 64
 * otherwise), the bf16 call's head counts; PKV_ERR_UNSUPPORTED when a batch's
 * per-sequence table and the kernel's stages do not fit in shared memory together
 * (about 2,200 sequences in a batch with prefill rows).
 */
int pkv_paged_attention_varlen_fp8(void *out, const void *q, const int32_t *query_start_loc,
                                   const void *k_cache, const void *v_cache,
                                   const int32_t *block_tables, const int32_t *context_lens,
                                   int num_seqs, int total_q_tokens, int max_q_len,
                                   int max_blocks_per_seq, int num_heads, int num_kv_heads,
                                   int head_dim, int block_size, int64_t num_blocks, float scale,
                                   int causal, float k_scale, float v_scale, void *workspace,
                                   size_t workspace_bytes, void *stream);

/*
 * Decode attention that allocates nothing and takes no workspace.  The pages have no
 * counterpart of this call: it exists for callers that are not allowed to allocate
 * device memory where they run attention -- e.g. a plugin executing inside another
 * runtime that reserved all device memory up front and forbids later allocations, or
 * a latency-critical loop that cannot afford cudaMalloc/cudaFree synchronizing the
 * device -- and that cannot thread a workspace buffer through to this call either.
 *
 * It computes exactly what pkv_paged_attention_decode computes, with the same
 * arguments minus the workspace.  Its scratch space is a fixed array of
 * PKV_STATIC_SCRATCH_BYTES inside the library's device image: every GPU on which the
 * library's kernels are loaded holds that array until the process exits.  Sizes whose
 * scratch would exceed it are refused with PKV_ERR_STATIC_SCRATCH_LIMIT before
 * anything is launched (pkv_workspace_size(PKV_OP_DECODE, ...) tells what a size
 * needs).  The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.  All calls on
 * a device share the one array and it keeps the previous call's contents (nothing in
 * it has to start at zero), so calls that can overlap on the GPU -- on different
 * streams, or from different host threads -- race and must not be issued.
 */
#define PKV_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
int pkv_paged_attention_decode_static(void *out, const void *q, const void *k_cache,
                                      const void *v_cache, const int32_t *block_tables,
                                      const int32_t *context_lens, int num_seqs,
                                      int max_blocks_per_seq, int num_heads, int num_kv_heads,
                                      int head_dim, int block_size, int64_t num_blocks,
                                      float scale, int dtype, void *stream);

/*
 * Step transfers: copies `bytes` bytes from host src to device dst (pkv_copy_to_device)
 * or from device src to host dst (pkv_copy_to_host), asynchronously on `stream`, in
 * stream order with the library's kernels.  When the host buffer is page-locked and
 * mapped into the device's address space (cudaHostAlloc, or cudaHostRegister with
 * mapping, on a unified-addressing system), the copy runs as a kernel whose threads load
 * or store the host memory directly (on GB300, over NVLink-C2C; for the few MB of a decode
 * step this is several times faster than a copy-engine transfer); otherwise it is a
 * cudaMemcpyAsync.  The device side must be memory of the current device
 * (PKV_ERR_INVALID_ARG otherwise).  Ownership stays with the caller; for a page-locked
 * host source the caller must not modify it until the copy has run.  Any alignment.
 * Not from the pages: the end-to-end step they describe moves its inputs and outputs
 * between host and device around the attention call.
 */
int pkv_copy_to_device(void *dst, const void *src, size_t bytes, void *stream);
int pkv_copy_to_host(void *dst, const void *src, size_t bytes, void *stream);

/*
 * Limit, in nanoseconds, of every pipeline wait inside the attention kernels launched
 * from now on (a consumer warp waiting for its K/V stage, a producer for a free stage).
 * A wait that runs out sets PKV_DEVERR_TIMEOUT, stops its CTA's pipeline, lets the
 * copies and tensor-core operations the CTA already issued complete, and the kernel
 * returns: the GPU context stays usable and pkv_get_device_error reports the flag.
 * Default 2 s (also restored by limit_ns = 0); a wait that ends normally takes
 * microseconds.  A short limit makes healthy launches give up too -- it exists so tests
 * can exercise the failure path.  Not from the pages.
 */
void pkv_set_wait_limit_ns(uint64_t limit_ns);

/*
 * Split-K of the decode rows for launches from now on (process-wide).  enabled != 0 (the
 * default): the blocks of all (sequence, KV-head tile) items are cut into equal shares,
 * one per CTA, and partial results are merged by log-sum-exp weights.  enabled == 0: every
 * item is computed whole by one CTA (each share boundary moves back to the first block of
 * the item it falls in; no merge work), the split's ablation: a long context then costs
 * one CTA's streaming time.  Results agree within rounding.  Not from the pages.
 */
void pkv_set_decode_split(int enabled);

/* Workspace bytes the op needs on the current device for these sizes (0 if the
 * sizes are unsupported).  Does not allocate. */
size_t pkv_workspace_size(int op, int num_seqs, int total_q_tokens, int num_heads,
                          int num_kv_heads, int head_dim, int block_size);

/* Static description of a status code. */
const char *pkv_status_string(int status);

/* Synchronizes `stream`, then returns and clears the current device's error word
 * (a bitwise OR of PKV_DEVERR_* flags; 0 = no error).  Negative on a CUDA error. */
int pkv_get_device_error(void *stream);

/*
 * Slot mapping on the host (step before the KV write).  [LESSON] "PagedAttention as
 * a virtual memory system": for new token t of sequence host_token_seq[t] at
 * absolute position p = host_token_pos[t]:
 *     host_slot_mapping[t] = host_block_tables[seq][p / block_size] * block_size
 *                            + p % block_size
 * host_token_seq[t] < 0 gives -1 (padding).  PKV_ERR_INVALID_ARG if p is negative,
 * beyond the table row, or lands on a negative table entry.
 */
int pkv_slot_mapping(int64_t *host_slot_mapping, const int32_t *host_block_tables,
                     int max_blocks_per_seq, const int32_t *host_token_seq,
                     const int32_t *host_token_pos, int64_t num_tokens, int block_size);

/*
 * Host block manager.  [LPNH] §2.2 BlockManager: a free list over num_blocks
 * physical block ids; allocate(n) takes the first n free ids or fails with
 * out-of-memory and changes nothing; free(ids) appends them to the list.  The
 * handle is host memory owned by the caller (create / destroy).  Not thread-safe.
 */
typedef struct pkv_block_manager pkv_block_manager;
pkv_block_manager *pkv_block_manager_create(int64_t num_blocks, int block_size);
void pkv_block_manager_destroy(pkv_block_manager *bm);
/* Writes n ids to host_ids_out; PKV_ERR_OOM (nothing taken) if fewer are free. */
int pkv_block_manager_allocate(pkv_block_manager *bm, int64_t n, int32_t *host_ids_out);
/* Drops one reference per listed id; a block whose last reference goes returns to the
 * tail of the free list (in the order listed).  PKV_ERR_INVALID_ARG (nothing changed)
 * if an id is outside the pool or listed more often than it is held. */
int pkv_block_manager_free(pkv_block_manager *bm, const int32_t *host_ids, int64_t n);
int64_t pkv_block_manager_num_free(const pkv_block_manager *bm);

/*
 * Shared read-only blocks ([LPNH] §4.3 prefix caching: requests with the same
 * system-prompt prefix reuse one set of read-only KV blocks).  A block allocated once
 * has one reference; share(ids) adds one reference per listed id (each must be held);
 * free drops one.  ref_count(id) returns the count (PKV_ERR_INVALID_ARG outside the
 * pool).  copy_on_write(id): the caller holds id and is about to write into it; if it is
 * the only holder, *host_new_id = id and 0 is returned (write in place); otherwise a
 * fresh block is taken from the free list, the caller's reference moves to it,
 * *host_new_id = the new id and 1 is returned -- the caller must then copy the block
 * on the device (pkv_copy_blocks) before writing.  PKV_ERR_OOM (nothing changed) if a
 * copy is needed and no block is free.
 */
int pkv_block_manager_share(pkv_block_manager *bm, const int32_t *host_ids, int64_t n);
int pkv_block_manager_ref_count(const pkv_block_manager *bm, int32_t id);
int pkv_block_manager_copy_on_write(pkv_block_manager *bm, int32_t id, int32_t *host_new_id);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
