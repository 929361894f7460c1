// paged_prefill.cu -- the plan of the chunked-prefill CTAs (tiles, shared-memory stages,
// workspace); their body is prefill_cta.cuh, run by paged_varlen_kernel (paged_varlen.cu).
#include "paged_prefill.cuh"

namespace pkv {

// ---- host side -------------------------------------------------------------------

int plan_prefill(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int sms,
                 int smem_optin, PrefillPlan *p, bool fp8) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads) return PKV_ERR_UNSUPPORTED;
    if (fp8 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    p->group = num_heads / num_kv_heads;
    if (p->group > 8) return PKV_ERR_UNSUPPORTED;
    // A tile is two halves of 16 * (8 / group) tokens x group heads (<= 128 rows each).
    p->tokens_per_tile = 2 * 16 * (8 / p->group);
    p->rows = p->tokens_per_tile * p->group;    // <= 256 rows per tile
    p->warps = kPrefillThreads / 32;  // producer, MMA issuer, 2 idle, a softmax warpgroup per half
    p->grid = sms < 256 ? sms : 256;  // the merge kernel holds <= 256 parts per tile
    p->max_seqs = num_seqs;
    const uint32_t q_bytes = (uint32_t)(head_dim / 64) * 2 * 128 * 128 + 8 * 4096;  // Q + epilogue staging
    p->stage_bytes = 128 * head_dim * 2;  // K or V of a 128-key chunk (16-bit operands)
    // barriers (11 + q_ready), TMEM slot and abort flag, scan scratch, per-sequence prefix
    const size_t fixed = 1024 + q_bytes + 8 * 12 + 8 + 32 * 8 + 8 * (size_t)(num_seqs + 1);
    const int64_t room = (int64_t)smem_optin - (int64_t)fixed;
    int nst, nst8 = 0;
    if (!fp8) {
        nst = (int)(room / (p->stage_bytes + 16));
        if (nst > 8) nst = 8;
    } else {
        // three fp16 operand slots (K of the next chunk loads while V of this one is read),
        // then as many e4m3 stages (128 keys x 128 bytes) as fit, up to 4
        nst = 3;
        const int64_t stage8 = 128 * head_dim;
        nst8 = (int)((room - 3 * (int64_t)(p->stage_bytes + 16)) / (stage8 + 16));
        if (nst8 > 4) nst8 = 4;
        if (nst8 < 1) return PKV_ERR_UNSUPPORTED;
    }
    if (nst < 3) return PKV_ERR_UNSUPPORTED;
    p->num_stages = nst;
    p->num_stages8 = nst8;
    p->smem = fixed + (size_t)nst * (p->stage_bytes + 16) + (size_t)nst8 * (128 * head_dim + 16);
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    p->off_jobs = 0;
    p->off_ml = up(sizeof(MergeJob) * (size_t)p->grid);
    p->off_o = p->off_ml + up(2 * (size_t)p->grid * p->rows * 8);
    p->ws_bytes = p->off_o + up(2 * (size_t)p->grid * p->rows * head_dim * 4);
    return PKV_OK;
}

}  // namespace pkv
