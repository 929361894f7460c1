// merge.cuh -- log-sum-exp merge of the parts of split work items.
//
// When a CTA share of the flat unit list starts or ends inside an item, each CTA that
// touched the item leaves a part in the workspace: per row its reference max m_p, sum
// l_p and unnormalised output o_p.  The softmax over the whole item is then
//     o = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p,   M = max_p m_p,
// which is exact: every part's weights are relative to its own m_p.
//
// The main kernel's CTA 0 writes one MergeJob per boundary between neighbouring CTA
// shares (the item split there, if that boundary is the item's first split); the merge
// kernel runs one thread per (row, 4 columns) of a job, so a job costs two rounds of global
// loads (the job; (m, l) and o of up to four parts together) and one more per four parts
// beyond.
#pragma once

#include "attn_block.cuh"
#include "pkv_split.cuh"

namespace pkv {

struct MergeJob {
    int64_t item_begin;   // first unit of the item
    int64_t total_units;  // T of the split
    int64_t out_row0;     // output row of the item's first token
    int32_t c0, c1;       // CTA shares holding its parts (c0 < c1); c0 < 0: no job
    int32_t ge;           // CTAs that took part in the split
    int32_t rows;         // live rows of the item
    int32_t rows_per_token;  // rows that share one output row (query heads per token)
    int32_t head0;        // query head of row 0
};

struct MergeArgs {
    const MergeJob *jobs;  // [grid]
    const float2 *ws_ml;   // [2 * grid][slot_rows]
    const float *ws_o;     // [2 * grid][slot_rows][head_dim]
    __nv_bfloat16 *out;
    int slot_rows;         // rows reserved per workspace slot
    int num_heads;
};

constexpr int kMergeMaxParts = 256;  // the grids hold <= 256 CTAs, so an item has <= 256 parts

__device__ __forceinline__ void no_job(MergeJob &j) {
    j.item_begin = j.total_units = j.out_row0 = 0;
    j.c0 = j.c1 = -1;
    j.ge = j.rows = j.rows_per_token = j.head0 = 0;
}

// One thread per (row, 4 columns) of a job; a CTA covers 256 / (D / 4) rows.  After the
// job (one load), every part's (m, l) and its 4 columns of o are loaded together, kPC
// parts per round, and combined in registers: o = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M)
// l_p, with M the running maximum over the rounds.  Two rounds of global loads for up to
// kPC parts, no shared memory and no CTA barrier.
template <int D>
__global__ void __launch_bounds__(256, 4) merge_parts_kernel(const MergeArgs m) {
    constexpr int CG = D / 4;         // 16-byte column groups of a row
    constexpr int RPC = 256 / CG;     // rows per CTA
    constexpr int kPC = 4;            // parts per round of loads
    pdl_wait();
    const MergeJob j = m.jobs[blockIdx.x];
    if (j.c0 < 0) return;
    const int nparts = j.c1 - j.c0 + 1;
    const int row = blockIdx.y * RPC + (int)threadIdx.x / CG;
    if (row >= j.rows || nparts > kMergeMaxParts) return;
    const int cg = (int)threadIdx.x % CG;
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = 0; p0 < nparts; p0 += kPC) {
        float2 ml[kPC];
        float4 o[kPC];
#pragma unroll
        for (int q = 0; q < kPC; ++q) {
            if (p0 + q < nparts) {
                const int slot = part_slot(j.c0 + p0 + q, j.item_begin, j.total_units, j.ge);
                const int64_t r = (int64_t)slot * m.slot_rows + row;
                ml[q] = __ldcg(m.ws_ml + r);
                o[q] = __ldcg(reinterpret_cast<const float4 *>(m.ws_o + r * D) + cg);
            } else {
                ml[q] = make_float2(-INFINITY, 0.f);
                o[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float mc = M;
#pragma unroll
        for (int q = 0; q < kPC; ++q) mc = fmaxf(mc, ml[q].x);
        if (mc == -INFINITY) continue;  // nothing seen yet (rows of empty parts keep weight 0)
        const float a0 = M == -INFINITY ? 0.f : fast_exp2(M - mc);
        L *= a0;
        acc.x *= a0;
        acc.y *= a0;
        acc.z *= a0;
        acc.w *= a0;
#pragma unroll
        for (int q = 0; q < kPC; ++q) {
            if (ml[q].x == -INFINITY) continue;
            const float w = fast_exp2(ml[q].x - mc);
            L += w * ml[q].y;
            acc.x += w * o[q].x;
            acc.y += w * o[q].y;
            acc.z += w * o[q].z;
            acc.w += w * o[q].w;
        }
        M = mc;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int tok = row / j.rows_per_token, hr = row - tok * j.rows_per_token;
    __nv_bfloat16 *orow = m.out + ((j.out_row0 + tok) * (int64_t)m.num_heads + j.head0 + hr) * D;
    uint2 packed;
    packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    reinterpret_cast<uint2 *>(orow)[cg] = packed;
}

template <int D>
cudaError_t launch_merge(const MergeArgs &m, int grid, cudaStream_t stream) {
    constexpr int RPC = 256 / (D / 4);
    const int ny = (m.slot_rows + RPC - 1) / RPC;
    return launch_pdl(merge_parts_kernel<D>, dim3(grid, ny), dim3(256), 0, stream, m);
}

}  // namespace pkv
