// fp8_block.cuh -- one warp's work on one 16-token block of an FP8 (e4m3) KV cache in the
// decode kernel: S^T = K Q^T and O^T += V^T P^T on m16n8k16 fp16 MMAs, with the e4m3 codes
// widened to fp16 (exactly) as the fragments are built.
//
// The block's K (or V) rows of one KV head sit in shared memory as 16 rows of 128
// bytes (head_dim 128, one e4m3 byte per element), written by TMA with 128-byte
// swizzling (16-byte chunk c of row r at chunk position c ^ (r % 8)).
//
// Both contractions are free to number their reduction index in any order, as long
// as the two operands agree; the numbering is chosen so that every thread reads whole
// 16-byte chunks instead of single bytes:
//  * S^T = K Q^T reduces over head dims.  In k-step ks, the fragment slots 2t, 2t+1,
//    2t+8, 2t+9 of thread t (t = lane % 4) hold dims 32t + 4ks + {0, 1, 2, 3}, so a
//    thread's K bytes for all 8 k-steps are the 32 contiguous bytes [32t, 32t + 32)
//    of its token rows, and its Q values the same 32 dims of its query heads.
//  * O^T += V^T P^T reduces over the block's tokens in their natural order and numbers
//    the head dims so that thread g (g = lane / 4) reads bytes [16g, 16g + 16) of four
//    token rows and its accumulators hold dims 16g .. 16g + 15 -- contiguous again when
//    the output is written.
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

// ---- heads on the MMA's N: the FP8 decode consumer ------------------------------------
//
// One warp, one KV head, up to 16 of its query heads, one 16-token block.  The tokens sit
// on the M of m16n8k16 fp16 MMAs and the query heads on N (8 per n-tile), so
//     S^T = K Q^T   (M = 16 tokens, N = heads, K = 128 dims: 8 MMAs per n-tile)
//     O^T += V^T P^T (M = 128 dims as 8 tiles of 16, N = heads, K = 16 tokens: 8 MMAs)
// -- half the MMAs of the heads-on-M form when a KV head has 8 query heads (rows 8..15 of
// that form were padding).  Lane (g, t) holds tokens g and g + 8 of heads 2t, 2t + 1 in S^T,
// and of O^T the dims 16g + 2mt (mt = 0..7, accumulator columns 0, 1) and 16g + 2mt + 1
// (columns 2, 3) of those heads.  QK^T reads bytes [32t, 32t + 32) of token rows g and
// g + 8, PV reads bytes [16g, 16g + 16) of token rows 2t, 2t + 1, 2t + 8, 2t + 9.  P^T
// reaches the B-operand layout with one movmatrix transpose per 8 x 8 half.

// NTH = n-tiles of query heads (1: up to 8 heads, 2: up to 16).
template <int NTH>
struct HeadState {
    float m[NTH][2], l[NTH][2];  // [n-tile][head 2t, 2t + 1]: reference max (base 2), partial sum
    float o[NTH][8][4];          // [n-tile][dim tile]: O^T accumulators
    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt) {
            m[nt][0] = m[nt][1] = -INFINITY;
            l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
        }
    }
};

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// S^T of the block for n-tile 0 (heads 0..7) and, if NTH = 2, 1 (heads 8..15); qa from
// load_q_fp8order (its rows g / g + 8 become the n-tiles' heads g).  s[nt][0..3] = heads
// (2t, 2t + 1) of token g, then of token g + 8.  Four accumulator chains per n-tile.
template <int NTH>
__device__ __forceinline__ void qk_block_fp8t(float (&s)[NTH][4], const uint32_t (&qa)[8][4], uint32_t tile,
                                              int lane) {
    const int g = lane >> 2, t = lane & 3;
    float c[NTH][4][4];
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int i = 0; i < 4; ++i) c[nt][k][i] = 0.f;
    uint32_t w[2][8];  // token rows g, g + 8: bytes [32t, 32t + 32)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int tok = h * 8 + g;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[h][0]), "=r"(w[h][1]), "=r"(w[h][2]), "=r"(w[h][3])
                     : "r"(tile + tok * 128 + (((2 * t) ^ (tok & 7)) << 4)));
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[h][4]), "=r"(w[h][5]), "=r"(w[h][6]), "=r"(w[h][7])
                     : "r"(tile + tok * 128 + (((2 * t + 1) ^ (tok & 7)) << 4)));
    }
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        uint32_t a[4];  // dims 32t + 4ks + {0, 1} (a0, a1) and {2, 3} (a2, a3) of tokens g, g + 8
        e4m3x4_to_f16x2x2(w[0][ks], a[0], a[2]);
        e4m3x4_to_f16x2x2(w[1][ks], a[1], a[3]);
        mma_f16_16816(c[0][ks & 3], a, qa[ks][0], qa[ks][2]);
        if constexpr (NTH == 2) mma_f16_16816(c[NTH - 1][ks & 3], a, qa[ks][1], qa[ks][3]);
    }
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[nt][i] = (c[nt][0][i] + c[nt][1][i]) + (c[nt][2][i] + c[nt][3][i]);
}

// Online softmax over the block's tokens for n-tile nt (scores scaled to base 2, -inf where
// masked), lazy rescale as in softmax_update (attn_block.cuh), fp16 weights (their row sum
// adds the fp32 values: fp16 keeps 11 significant bits); returns P^T as the PV B
// fragment pb[0..1] (tokens 2t, 2t + 1 / 2t + 8, 2t + 9 of head g).
template <int NTH>
__device__ __forceinline__ void softmax_update_t(HeadState<NTH> &st, int nt, const float (&s)[4], uint32_t (&pb)[2]) {
    float mA = fmaxf(s[0], s[2]), mB = fmaxf(s[1], s[3]);  // heads 2t, 2t + 1
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, off));
        mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, off));
    }
    const bool upA = mA > st.m[nt][0] + kRescaleSlack;  // false while the max is -inf
    const bool upB = mB > st.m[nt][1] + kRescaleSlack;
    if (__any_sync(0xffffffffu, upA || upB)) {
        const float aA = upA ? fast_exp2(st.m[nt][0] - mA) : 1.f;
        const float aB = upB ? fast_exp2(st.m[nt][1] - mB) : 1.f;
        if (upA) st.m[nt][0] = mA;
        if (upB) st.m[nt][1] = mB;
        st.l[nt][0] *= aA;
        st.l[nt][1] *= aB;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            st.o[nt][mt][0] *= aA;
            st.o[nt][mt][2] *= aA;
            st.o[nt][mt][1] *= aB;
            st.o[nt][mt][3] *= aB;
        }
    }
    const float bA = st.m[nt][0] == -INFINITY ? 0.f : st.m[nt][0];
    const float bB = st.m[nt][1] == -INFINITY ? 0.f : st.m[nt][1];
    const float eA0 = fast_exp2(s[0] - bA), eB0 = fast_exp2(s[1] - bB);  // token g
    const float eA1 = fast_exp2(s[2] - bA), eB1 = fast_exp2(s[3] - bB);  // token g + 8
    st.l[nt][0] += eA0 + eA1;
    st.l[nt][1] += eB0 + eB1;
    pb[0] = movmatrix_trans(pack_f16x2(eA0, eB0));  // tokens 0..7 x heads 0..7, transposed
    pb[1] = movmatrix_trans(pack_f16x2(eA1, eB1));  // tokens 8..15
}

// O^T += V^T P^T for the block (V in e4m3 codes; the V scale is applied when the output is
// written).  Token rows at or past `valid` are zeroed before use (the pool there may hold
// NaN codes).
template <bool MASKED, int NTH>
__device__ __forceinline__ void pv_block_fp8t(HeadState<NTH> &st, const uint32_t (&pb)[NTH][2], uint32_t tile,
                                              int valid, int lane) {
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
            // dim tile mt = 2w + b / 2: dims 16g + 2mt (rows g) and 16g + 2mt + 1 (rows g + 8)
            const uint32_t sel = (uint32_t)b | ((4u + b) << 4) | ((b + 1u) << 8) | ((5u + b) << 12);
            const uint32_t lo = __byte_perm(r[0][w], r[1][w], sel);  // tokens 2t, 2t + 1
            const uint32_t hi = __byte_perm(r[2][w], r[3][w], sel);  // tokens 2t + 8, 2t + 9
            uint32_t a[4];
            e4m3x4_to_f16x2x2(lo, a[0], a[1]);
            e4m3x4_to_f16x2x2(hi, a[2], a[3]);
            const int mt = 2 * w + b / 2;
#pragma unroll
            for (int nt = 0; nt < NTH; ++nt) mma_f16_16816(st.o[nt][mt], a, pb[nt][0], pb[nt][1]);
        }
    }
}

// The partial sums across the 8 lanes that share t (each held tokens g, g + 8).
template <int NTH>
__device__ __forceinline__ void finish_sums_t(HeadState<NTH> &st) {
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) st.l[nt][e] += __shfl_xor_sync(0xffffffffu, st.l[nt][e], off);
}

}  // namespace pkv
