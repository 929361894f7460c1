// fp8_block.cuh -- one warp's work on one 16-token block of an FP8 (e4m3) KV cache:
// S = Q K^T and O += P V on m16n8k16 fp16 MMAs, with the e4m3 codes widened to fp16
// (exactly) as the fragments are built.
//
// The block's K (or V) rows of one KV head sit in shared memory as 16 rows of 128
// bytes (head_dim 128, one e4m3 byte per element), written by TMA with 128-byte
// swizzling (16-byte chunk c of row r at chunk position c ^ (r % 8)).
//
// Both contractions are free to number their reduction index in any order, as long
// as the two operands agree; the numbering below is chosen so that every thread reads
// whole 16-byte chunks instead of single bytes:
//  * S = Q K^T reduces over head dims.  In k-step ks, the fragment slots 2t, 2t+1,
//    2t+8, 2t+9 of thread t (t = lane % 4) hold dims 32t + 4ks + {0, 1, 2, 3}, so a
//    thread's K bytes for all 8 k-steps are the 32 contiguous bytes [32t, 32t + 32)
//    of its key row, and its Q values the same 32 dims of its query rows.
//  * O += P V reduces over the block's tokens in their natural order (P comes
//    straight from the S accumulators) and produces head dims in the order
//    "n-tile j, column n holds dim 16n + j": thread g (g = lane / 4) reads bytes
//    [16g, 16g + 16) of four token rows, and its accumulators hold dims 32t + j and
//    32t + 16 + j -- contiguous runs again when the output is written.
#pragma once

#include <cuda_fp16.h>

#include "attn_block.cuh"

namespace pkv {

// Four e4m3 codes (one 32-bit word, lowest byte first) -> two fp16x2 words: lo holds
// bytes 0, 1 and hi bytes 2, 3 (lower byte in the lower half); exact.  The word's 16-bit
// halves feed the conversions directly, with no masking or shifting.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// Two bf16 (one 32-bit word, low half first) -> two fp16, round to nearest even.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    const __half2 h = __floats2half2_rn(bf16_lo(w), bf16_hi(w));
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Q fragments (A operand, fp16) of the warp's 16 query rows in the k numbering above.
// q0 points at the row of query head r0; rows at or past rows_valid read as zero.
__device__ __forceinline__ void load_q_fp8order(uint32_t (&qa)[8][4], const __nv_bfloat16 *q0, int rows_valid,
                                                int lane) {
    const int g = lane >> 2, t = lane & 3;
    uint32_t w0[16], w1[16];  // rows g and g + 8, dims [32t, 32t + 32) as bf16 pairs
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 a = make_uint4(0u, 0u, 0u, 0u), b = make_uint4(0u, 0u, 0u, 0u);
        if (g < rows_valid) a = __ldg(reinterpret_cast<const uint4 *>(q0 + g * 128 + 32 * t) + i);
        if (g + 8 < rows_valid) b = __ldg(reinterpret_cast<const uint4 *>(q0 + (g + 8) * 128 + 32 * t) + i);
        w0[4 * i] = a.x; w0[4 * i + 1] = a.y; w0[4 * i + 2] = a.z; w0[4 * i + 3] = a.w;
        w1[4 * i] = b.x; w1[4 * i + 1] = b.y; w1[4 * i + 2] = b.z; w1[4 * i + 3] = b.w;
    }
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        qa[ks][0] = bf16x2_to_f16x2(w0[2 * ks]);      // dims 32t + 4ks + {0, 1}, row g
        qa[ks][1] = bf16x2_to_f16x2(w1[2 * ks]);      // row g + 8
        qa[ks][2] = bf16x2_to_f16x2(w0[2 * ks + 1]);  // dims 32t + 4ks + {2, 3}
        qa[ks][3] = bf16x2_to_f16x2(w1[2 * ks + 1]);
    }
}

// S (16 rows x 16 tokens, fp32) = Q K^T (K in e4m3 codes; the K scale is applied to S
// by the caller).  Eight accumulator chains of two MMAs each (k-steps ks and ks + 4 of one
// n-tile share a chain): the legacy MMA's latency, not its issue rate, bounds this loop.
__device__ __forceinline__ void qk_block_fp8(float (&s)[2][4], const uint32_t (&qa)[8][4], uint32_t tile, int lane) {
    const int g = lane >> 2, t = lane & 3;
    float c[2][4][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int i = 0; i < 4; ++i) c[nt][k][i] = 0.f;
    uint32_t w[2][8];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int tok = nt * 8 + g;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[nt][0]), "=r"(w[nt][1]), "=r"(w[nt][2]), "=r"(w[nt][3])
                     : "r"(tile + tok * 128 + (((2 * t) ^ (tok & 7)) << 4)));
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[nt][4]), "=r"(w[nt][5]), "=r"(w[nt][6]), "=r"(w[nt][7])
                     : "r"(tile + tok * 128 + (((2 * t + 1) ^ (tok & 7)) << 4)));
    }
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            uint32_t b0, b1;  // dims 32t + 4ks + {0, 1} and {2, 3}
            e4m3x4_to_f16x2x2(w[nt][ks], b0, b1);
            mma_f16_16816(c[nt][ks & 3], qa[ks], b0, b1);
        }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[nt][i] = (c[nt][0][i] + c[nt][1][i]) + (c[nt][2][i] + c[nt][3][i]);
}

// O += P V for one block (V in e4m3 codes; the V scale is applied by the caller when the
// output is written).  o[j] collects head dims 32t + j (columns 0, 2) and 32t + 16 + j
// (columns 1, 3).  Token rows at or past `valid` are zeroed before use (the pool there
// may hold NaN codes).
template <bool MASKED>
__device__ __forceinline__ void pv_block_fp8(float (&o)[16][4], const uint32_t (&pa)[4], uint32_t tile, int valid,
                                             int lane) {
    const int g = lane >> 2, t = lane & 3;
    uint32_t r[4][4];  // token rows 2t, 2t + 1, 2t + 8, 2t + 9; bytes [16g, 16g + 16)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int tok = 2 * t + (i & 1) + 8 * (i >> 1);
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[i][0]), "=r"(r[i][1]), "=r"(r[i][2]), "=r"(r[i][3])
                     : "r"(tile + tok * 128 + ((g ^ (tok & 7)) << 4)));
        if (MASKED && tok >= valid) r[i][0] = r[i][1] = r[i][2] = r[i][3] = 0u;
    }
#pragma unroll
    for (int w = 0; w < 4; ++w) {
#pragma unroll
        for (int b = 0; b < 4; b += 2) {
            // bytes (row 2t, row 2t+1) of dims 16g + 4w + b and + 1, and the same for
            // rows 2t+8, 2t+9: the k pairs of the B fragment for n-tiles 4w + b, 4w + b + 1
            const uint32_t sel = (uint32_t)b | ((4u + b) << 4) | ((b + 1u) << 8) | ((5u + b) << 12);
            const uint32_t lo = __byte_perm(r[0][w], r[1][w], sel);
            const uint32_t hi = __byte_perm(r[2][w], r[3][w], sel);
            const int j = 4 * w + b;
            uint32_t lo0, lo1, hi0, hi1;
            e4m3x4_to_f16x2x2(lo, lo0, lo1);
            e4m3x4_to_f16x2x2(hi, hi0, hi1);
            mma_f16_16816(o[j], pa, lo0, hi0);
            mma_f16_16816(o[j + 1], pa, lo1, hi1);
        }
    }
}

}  // namespace pkv
