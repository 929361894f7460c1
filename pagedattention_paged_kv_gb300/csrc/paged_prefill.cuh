// paged_prefill.cuh -- arguments and plan of the chunked-prefill CTAs (prefill_cta.cuh,
// paged_prefill.cu): attention for every sequence of a varlen batch with q_len >= 2.
#pragma once

#include "merge.cuh"
#include "pkv_common.cuh"

namespace pkv {

// 12 warps: warpgroup 0 = TMA producer, tcgen05 issuer and two warps that convert FP8
// operands (idle with a bf16 cache); warpgroups 1 and 2 = softmax of the tile's two
// halves.  Launched at 168 registers a thread, the most 12 warps may hold.
constexpr int kPrefillThreads = 384;

// A work item ("tile") is tokens_per_tile consecutive query tokens of one sequence
// together with all `group` query heads of one KV head: rows r = token * group + head,
// at most 16 * max_warps rows.  Its units are the 16-token key blocks it must visit.
struct PrefillArgs {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *q;
    const int32_t *query_start_loc;
    const int32_t *block_tables;
    const int32_t *context_lens;
    int total_q;  // rows of q and out
    int num_seqs;
    int max_blocks_per_seq;
    int num_heads;
    int num_kv_heads;
    int group;
    int tokens_per_tile;  // a multiple of 16
    int grid;
    int num_stages;
    bool causal;
    int64_t num_blocks;
    float scale_log2;
    MergeJob *ws_jobs;       // [grid]
    float2 *ws_ml;           // [2 * grid][rows]
    float *ws_o;             // [2 * grid][rows][head_dim]
    int max_seqs;
    int *err;
    uint64_t wait_ns;  // limit of a pipeline wait (see pkv_common.cuh)
    // FP8 cache (the FP8 kernel): e4m3 K/V land in a ring of num_stages8 byte stages and are
    // widened to fp16 into the num_stages-slot operand ring; V elements mean code x v_scale
    // (the K scale is folded into scale_log2).
    int num_stages8;
    float v_scale;
};

struct PrefillPlan {
    int group, tokens_per_tile, rows, warps, grid, num_stages, stage_bytes, max_seqs, num_stages8;
    size_t smem;
    size_t off_jobs, off_ml, off_o, ws_bytes;
};

// Fills *p for these sizes (num_seqs bounds the per-sequence table); PKV_OK or
// PKV_ERR_UNSUPPORTED.
int plan_prefill(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int sms,
                 int smem_optin, PrefillPlan *p, bool fp8 = false);

}  // namespace pkv
