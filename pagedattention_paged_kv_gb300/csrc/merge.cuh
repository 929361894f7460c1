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
// kernel runs one CTA per 16 rows of a job, so a job costs three rounds of global loads
// (job, (m, l) of its parts, o of its parts) whatever the batch and however many parts.
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

constexpr int kMergeRows = 16;       // rows per CTA; a job gets ceil(slot_rows / 16) CTAs
constexpr int kMergeMaxParts = 256;  // the grids hold <= 256 CTAs, so an item has <= 256 parts

__device__ __forceinline__ void no_job(MergeJob &j) {
    j.item_begin = j.total_units = j.out_row0 = 0;
    j.c0 = j.c1 = -1;
    j.ge = j.rows = j.rows_per_token = j.head0 = 0;
}

// Three rounds of global loads per CTA (the job; (m, l) of its rows' parts; o of its
// rows' parts).  The 8 warps split the (row, part) pairs: G = min(8, parts) part groups
// (a power of two) times 8 / G row groups, so a job split into many parts keeps every warp
// busy with independent loads and a two-part job still uses all warps.  The part groups'
// sums are added in group order (bit-reproducible).
template <int D>
__global__ void __launch_bounds__(256, 4) merge_parts_kernel(const MergeArgs m) {
    constexpr int D4 = D / 4;
    __shared__ float s_w[kMergeRows][kMergeMaxParts];  // m_p, then the weight 2^(m_p - M)
    __shared__ float s_inv[kMergeRows];
    __shared__ float4 s_acc[kMergeRows][D4];
    pdl_wait();
    const MergeJob j = m.jobs[blockIdx.x];
    if (j.c0 < 0) return;
    const int nparts = j.c1 - j.c0 + 1;
    const int row0 = blockIdx.y * kMergeRows;
    if (row0 >= j.rows || nparts > kMergeMaxParts) return;
    const int nrows = min(kMergeRows, j.rows - row0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // (1) warp w: the weights of rows w and w + 8
    for (int k = warp; k < nrows; k += 8) {
        const int row = row0 + k;
        float M = -INFINITY, lv[kMergeMaxParts / 32];
#pragma unroll
        for (int i = 0; i < kMergeMaxParts / 32; ++i) {
            const int p = lane + 32 * i;
            lv[i] = 0.f;
            if (p < nparts) {
                const int slot = part_slot(j.c0 + p, j.item_begin, j.total_units, j.ge);
                const float2 ml = m.ws_ml[(int64_t)slot * m.slot_rows + row];
                s_w[k][p] = ml.x;
                lv[i] = ml.y;
                M = fmaxf(M, ml.x);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float base = M == -INFINITY ? 0.f : M;  // rows that saw nothing keep weight 0
        float L = 0.f;
#pragma unroll
        for (int i = 0; i < kMergeMaxParts / 32; ++i) {
            const int p = lane + 32 * i;
            if (p < nparts) {
                const float w = fast_exp2(s_w[k][p] - base);
                s_w[k][p] = w;
                L += w * lv[i];
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (lane == 0) s_inv[k] = 1.f / L;
    }
    __syncthreads();
    // (2) warp w = (row group rg, part group pg): rows rg, rg + RG, ...; parts pg, pg + G, ...
    const int G = nparts >= 8 ? 8 : nparts >= 4 ? 4 : nparts >= 2 ? 2 : 1;
    const int RG = 8 / G;
    const int pg = warp % G, rg = warp / G;
    static_assert(D4 <= 32, "one lane per 4 columns");
    const int d4 = lane;
    const bool col = d4 < D4;
    // rows in passes of 4 per warp (few registers: the CTA then fits next to the tail of
    // the kernel that produced the parts)
    for (int r0 = 0; r0 < nrows; r0 += 4 * RG) {
        float4 acc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (col) {
#pragma unroll 2
            for (int p = pg; p < nparts; p += G) {
                const int slot = part_slot(j.c0 + p, j.item_begin, j.total_units, j.ge);
                const float4 *ob =
                    reinterpret_cast<const float4 *>(m.ws_o + ((int64_t)slot * m.slot_rows + row0) * D);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int k = r0 + rg + i * RG;
                    if (k < nrows) {
                        const float w = s_w[k][p];
                        const float4 ov = ob[k * D4 + d4];
                        acc[i].x += w * ov.x;
                        acc[i].y += w * ov.y;
                        acc[i].z += w * ov.z;
                        acc[i].w += w * ov.w;
                    }
                }
            }
        }
        // (3) add the part groups in order: group 0 stores, groups 1 .. G-1 add in turn
        // (every thread takes every barrier)
        for (int g = 0; g < G; ++g) {
            if (pg == g && col) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int k = r0 + rg + i * RG;
                    if (k < nrows) {
                        if (g == 0) {
                            s_acc[k][d4] = acc[i];
                        } else {
                            float4 t = s_acc[k][d4];
                            t.x += acc[i].x;
                            t.y += acc[i].y;
                            t.z += acc[i].z;
                            t.w += acc[i].w;
                            s_acc[k][d4] = t;
                        }
                    }
                }
            }
            __syncthreads();
        }
    }
    // (4) one thread per (row, 4 columns): normalise, store bf16
    for (int idx = threadIdx.x; idx < nrows * D4; idx += blockDim.x) {
        const int k = idx / D4, d4 = idx - k * D4;
        const float4 t = s_acc[k][d4];
        const float inv = s_inv[k];
        const int row = row0 + k;
        const int tok = row / j.rows_per_token, hr = row - tok * j.rows_per_token;
        __nv_bfloat16 *orow = m.out + ((j.out_row0 + tok) * (int64_t)m.num_heads + j.head0 + hr) * D;
        uint2 packed;
        packed.x = pack_bf16x2(t.x * inv, t.y * inv);
        packed.y = pack_bf16x2(t.z * inv, t.w * inv);
        reinterpret_cast<uint2 *>(orow)[d4] = packed;
    }
}

template <int D>
cudaError_t launch_merge(const MergeArgs &m, int grid, cudaStream_t stream) {
    const int ny = (m.slot_rows + kMergeRows - 1) / kMergeRows;
    return launch_pdl(merge_parts_kernel<D>, dim3(grid, ny), dim3(256), 0, stream, m);
}

}  // namespace pkv
