// bf16t_block.cuh -- one warp's work on one 16-token block of a bf16 KV cache in the decode
// kernel, with the query heads on the N of m16n8k16 bf16 MMAs (the form fp8_block.cuh uses
// for an FP8 cache):
//     S^T = K Q^T    (M = the block's 16 tokens, N = 8 query heads, K = head dims)
//     O^T += V^T P^T (M = head dims in tiles of 16, N = the heads, K = the 16 tokens)
// A KV head with 8 query heads fills N exactly, where the heads-on-M form (attn_block.cuh)
// pads M = 16 with 8 empty rows: half the MMAs, and a shorter chain per block.
//
// K (or V) of the block sits in shared memory as [head_dim / 64] sub-tiles of [16 tokens][64]
// bf16, written by TMA with 128-byte swizzling.  K's tile is the A operand as it stands
// (ldmatrix); V's tile, read transposed (ldmatrix.trans), is V^T.  Lane (g, t) = (lane / 4,
// lane % 4) holds S^T of tokens g and g + 8 for heads 2t, 2t + 1, and of O^T the dims
// 16mt + g and 16mt + g + 8 of those heads.  The softmax state is fp8_block.cuh's HeadState;
// its weights here are bf16 and its row sums add exactly those rounded weights (so a
// one-token context returns V exactly).
#pragma once

#include "fp8_block.cuh"

namespace pkv {

// Q^T fragments (B operand) of the warp's heads: n-tile nt holds heads 8nt .. 8nt + 7 of the
// warp's 16 (q0 points at head r0); qb[nt][ks] = dims 16ks + 2t, +1 and 16ks + 2t + 8, +9 of
// head 8nt + g.  Heads at or past rows_valid read as zero.
template <int D, int NTH>
__device__ __forceinline__ void load_q_bt(uint32_t (&qb)[NTH][D / 16][2], const __nv_bfloat16 *q0, int rows_valid,
                                          int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt) {
        const bool ok = 8 * nt + g < rows_valid;
        const uint32_t *row = reinterpret_cast<const uint32_t *>(q0 + (int64_t)(8 * nt + g) * D);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qb[nt][ks][0] = ok ? __ldg(row + (16 * ks + 2 * t) / 2) : 0u;
            qb[nt][ks][1] = ok ? __ldg(row + (16 * ks + 2 * t + 8) / 2) : 0u;
        }
    }
}

// S^T of the block: s[nt][0..3] = heads (2t, 2t + 1) of token g, then of token g + 8.  Four
// accumulator chains per n-tile.
template <int D, int NTH>
__device__ __forceinline__ void qk_block_bt(float (&s)[NTH][4], const uint32_t (&qb)[NTH][D / 16][2],
                                            uint32_t tile, uint32_t chunk_stride, int lane) {
    float c[NTH][4][4];
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int i = 0; i < 4; ++i) c[nt][k][i] = 0.f;
    // matrices of the 16 x 16 A tile: (tokens 0-7, dims 0-7), (8-15, 0-7), (0-7, 8-15), (8-15, 8-15)
    const int mat = lane >> 3, r = lane & 7;
    const int tok = ((mat & 1) << 3) + r;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const int col = ks * 16 + ((mat >> 1) << 3);
        uint32_t a[4];
        ldmatrix_x4(tile + (col >> 6) * chunk_stride + swz128(tok, col & 63), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt) mma_bf16_16816(c[nt][ks & 3], a, qb[nt][ks][0], qb[nt][ks][1]);
    }
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) s[nt][i] = (c[nt][0][i] + c[nt][1][i]) + (c[nt][2][i] + c[nt][3][i]);
}

// Online softmax over the block's tokens for n-tile nt (scores scaled to base 2, -inf where
// masked), the lazy rescale of softmax_update (attn_block.cuh); bf16 weights, whose rounded
// values the row sums add; returns P^T as the PV B fragment pb[0..1] (tokens 2t, 2t + 1 /
// 2t + 8, 2t + 9 of head g).
template <int NTH>
__device__ __forceinline__ void softmax_update_bt(HeadState<NTH> &st, int nt, const float (&s)[4], uint32_t (&pb)[2]) {
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
    const uint32_t p0 = pack_bf16x2(fast_exp2(s[0] - bA), fast_exp2(s[1] - bB));  // token g: heads 2t, 2t + 1
    const uint32_t p1 = pack_bf16x2(fast_exp2(s[2] - bA), fast_exp2(s[3] - bB));  // token g + 8
    st.l[nt][0] += bf16_lo(p0) + bf16_lo(p1);
    st.l[nt][1] += bf16_hi(p0) + bf16_hi(p1);
    pb[0] = movmatrix_trans(p0);  // tokens 0..7 x heads 0..7, transposed
    pb[1] = movmatrix_trans(p1);  // tokens 8..15
}

// O^T += V^T P^T for the block; V rows at or past `valid` are zeroed in the fragments (the
// pool there may hold NaN).  MASKED = false skips the zeroing when all 16 rows count.
template <int D, bool MASKED, int NTH>
__device__ __forceinline__ void pv_block_bt(HeadState<NTH> &st, const uint32_t (&pb)[NTH][2], uint32_t tile,
                                            uint32_t chunk_stride, int valid, int lane) {
    const int t = lane & 3;
    uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;  // tokens 2t, 2t + 1 / 2t + 8, 2t + 9
    if (MASKED) {
        keep_lo = (2 * t < valid ? 0x0000ffffu : 0u) | (2 * t + 1 < valid ? 0xffff0000u : 0u);
        keep_hi = (8 + 2 * t < valid ? 0x0000ffffu : 0u) | (8 + 2 * t + 1 < valid ? 0xffff0000u : 0u);
    }
    // matrices of V^T's 16 x 16 A tile, each read transposed from V: (tokens 0-7, dims 0-7),
    // (tokens 0-7, dims 8-15), (tokens 8-15, dims 0-7), (tokens 8-15, dims 8-15)
    const int mat = lane >> 3, r = lane & 7;
    const int tok = ((mat >> 1) << 3) + r;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        const int col = mt * 16 + ((mat & 1) << 3);
        uint32_t a[4];
        ldmatrix_x4_trans(tile + (col >> 6) * chunk_stride + swz128(tok, col & 63), a[0], a[1], a[2], a[3]);
        if (MASKED) {
            a[0] &= keep_lo;
            a[1] &= keep_lo;
            a[2] &= keep_hi;
            a[3] &= keep_hi;
        }
#pragma unroll
        for (int nt = 0; nt < NTH; ++nt) mma_bf16_16816(st.o[nt][mt], a, pb[nt][0], pb[nt][1]);
    }
}

}  // namespace pkv
