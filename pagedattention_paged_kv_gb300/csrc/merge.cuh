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
// kernel runs one CTA row-slice per job, so a job costs three rounds of global loads
// (job, (m, l) of its parts, o of its parts) whatever the batch.
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

constexpr int kMergeMaxRows = 16;    // rows per CTA; a job gets ceil(slot_rows / 16) CTAs
constexpr int kMergeSmemParts = 32;  // parts whose (m, l) and weight stay in shared memory

__device__ __forceinline__ void no_job(MergeJob &j) {
    j.item_begin = j.total_units = j.out_row0 = 0;
    j.c0 = j.c1 = -1;
    j.ge = j.rows = j.rows_per_token = j.head0 = 0;
}

template <int D>
__global__ void __launch_bounds__(256) merge_parts_kernel(const MergeArgs m) {
    __shared__ float2 s_ml[kMergeMaxRows][kMergeSmemParts];
    __shared__ float s_base[kMergeMaxRows], s_inv[kMergeMaxRows];
    pdl_wait();
    const MergeJob j = m.jobs[blockIdx.x];
    if (j.c0 < 0) return;
    const int nparts = j.c1 - j.c0 + 1;
    const int np_s = nparts < kMergeSmemParts ? nparts : kMergeSmemParts;
    const int y = blockIdx.y, ny = gridDim.y;  // rows y, y + ny, y + 2 ny, ...
    const int my_rows = (j.rows - y + ny - 1) / ny;
    if (my_rows <= 0) return;
    // (m, l) of my rows x the first parts, all loads in flight together
    for (int i = threadIdx.x; i < my_rows * np_s; i += blockDim.x) {
        const int k = i / np_s, p = i - k * np_s;
        const int slot = part_slot(j.c0 + p, j.item_begin, j.total_units, j.ge);
        s_ml[k][p] = m.ws_ml[(int64_t)slot * m.slot_rows + y + k * ny];
    }
    __syncthreads();
    for (int k = threadIdx.x; k < my_rows; k += blockDim.x) {
        const int row = y + k * ny;
        float M = -INFINITY;
        for (int p = 0; p < nparts; ++p)
            M = fmaxf(M, p < np_s ? s_ml[k][p].x
                                  : m.ws_ml[(int64_t)part_slot(j.c0 + p, j.item_begin, j.total_units, j.ge) *
                                                m.slot_rows + row].x);
        const float base = M == -INFINITY ? 0.f : M;  // rows that saw nothing keep weight 0
        float L = 0.f;
        for (int p = 0; p < nparts; ++p) {
            const float2 ml = p < np_s ? s_ml[k][p]
                                       : m.ws_ml[(int64_t)part_slot(j.c0 + p, j.item_begin, j.total_units, j.ge) *
                                                     m.slot_rows + row];
            const float w = fast_exp2(ml.x - base);
            L += w * ml.y;
            if (p < np_s) s_ml[k][p].x = w;  // keep the weight in place of m
        }
        s_base[k] = base;
        s_inv[k] = 1.f / L;
    }
    __syncthreads();
    constexpr int D4 = D / 4;
    for (int task = threadIdx.x; task < my_rows * D4; task += blockDim.x) {
        const int k = task / D4, d4 = task - k * D4;
        const int row = y + k * ny;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int p = 0; p < nparts; ++p) {
            const int slot = part_slot(j.c0 + p, j.item_begin, j.total_units, j.ge);
            const float w = p < np_s ? s_ml[k][p].x
                                     : fast_exp2(m.ws_ml[(int64_t)slot * m.slot_rows + row].x - s_base[k]);
            const float4 ov = reinterpret_cast<const float4 *>(m.ws_o + ((int64_t)slot * m.slot_rows + row) * D)[d4];
            acc.x += w * ov.x;
            acc.y += w * ov.y;
            acc.z += w * ov.z;
            acc.w += w * ov.w;
        }
        const float inv = s_inv[k];
        const int tok = row / j.rows_per_token, hr = row - tok * j.rows_per_token;
        __nv_bfloat16 *orow =
            m.out + ((j.out_row0 + tok) * (int64_t)m.num_heads + j.head0 + hr) * D;
        uint2 packed;
        packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        reinterpret_cast<uint2 *>(orow)[d4] = packed;
    }
}

template <int D>
cudaError_t launch_merge(const MergeArgs &m, int grid, cudaStream_t stream) {
    const int ny = (m.slot_rows + kMergeMaxRows - 1) / kMergeMaxRows;
    return launch_pdl(merge_parts_kernel<D>, dim3(grid, ny), dim3(256), 0, stream, m);
}

}  // namespace pkv
