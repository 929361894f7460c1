// paged_decode.cuh -- arguments and launcher of the decode kernel (paged_decode.cu).
#pragma once

#include "merge.cuh"
#include "pkv_common.cuh"

namespace pkv {

// Everything the decode kernel and its merge kernel read.  A work item ("virtual
// sequence") is one (sequence, tile of heads_per_cta KV heads); item v = s *
// head_tiles + tile.
struct DecodeArgs {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *q;
    const int32_t *block_tables;
    const int32_t *context_lens;
    const int32_t *query_start_loc;  // null: decode (row s); else only q_len == 1 sequences
    int total_q;                     // rows of q and out
    int num_seqs;
    int max_blocks_per_seq;
    int block_size;      // tokens per pool block: 8, 16, 32 or 64
    int num_heads;
    int group;           // num_heads / num_kv_heads
    int heads_per_cta;   // KV heads per work item
    int head_tiles;      // num_kv_heads / heads_per_cta
    int warps_per_head;  // ceil(group / 16)
    int num_stages;      // shared-memory ring depth (K and V of a block take one stage each)
    int grid;            // CTAs launched
    int min_blocks_per_cta;
    int whole_items;     // 1: no item is split across CTAs (shares end at item boundaries)
    int64_t num_blocks;
    float scale_log2;    // scale * log2(e) (times the K scale for an FP8 cache)
    float v_scale;       // FP8 cache: V element = code value * v_scale (1 otherwise)
    MergeJob *ws_jobs;   // [grid]
    float2 *ws_ml;       // [2 * grid][heads_per_cta * group]  (running max, sum)
    float *ws_o;         // [2 * grid][heads_per_cta * group][head_dim]
    int *err;            // device error word
    uint64_t wait_ns;    // limit of a pipeline wait (see pkv_common.cuh)
    // Fused KV write (null k_new: none): before a sequence's last unit is read, its new
    // token's rows k_new[s], v_new[s] ([num_seqs][Hkv][D] bf16) are stored at position
    // context_lens[s] - 1 of k_cache_w / v_cache_w (quantised with k_scale_q / v_scale_q for
    // an FP8 cache).
    const void *k_new;
    const void *v_new;
    void *k_cache_w;
    void *v_cache_w;
    float k_scale_q;
    float v_scale_q;
};

size_t decode_smem_bytes(int stage_bytes, int num_stages, int num_items);
cudaError_t launch_paged_decode(int head_dim, bool fp8, const CUtensorMap &k_map, const CUtensorMap &v_map,
                                const DecodeArgs &a, size_t smem, cudaStream_t stream);

}  // namespace pkv
