// attn_block.cuh -- one warp's work on one 16-token KV block: S = Q K^T, the online
// softmax update, O += P V.  Shared by the decode and the chunked-prefill kernels.
//
// A warp owns 16 query rows (the M of an m16n8k16 bf16 MMA).  K and V of the block
// sit in shared memory as [head_dim / 64] sub-tiles of [16 tokens][64] bf16, written by
// TMA with 128-byte swizzling; `tile` is the first sub-tile's shared address and
// `chunk_stride` the distance between sub-tiles.
#pragma once

#include <atomic>

#include <cuda_fp16.h>

#include "pkv_common.cuh"

namespace pkv {

// Running softmax state of the lane's two rows (g and g + 8 of the warp's 16):
// reference max m (base-2 units), sum l of exp2(s - m), and O = sum exp2(s - m) V.
template <int D>
struct RowState {
    float m0, m1, l0, l1;
    float o[D / 8][4];
    __device__ __forceinline__ void reset() {
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    }
};

// S (16 rows x 16 tokens, fp32) = Q K^T.  Four independent accumulator chains (two
// per 8-token half, even and odd k-steps) keep the MMA dependency chains short.
template <int D>
__device__ __forceinline__ void qk_block(float (&s)[2][4], const uint32_t (&qa)[D / 16][4],
                                         uint32_t tile, uint32_t chunk_stride, int lane) {
    float t[2][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) s[0][i] = s[1][i] = t[0][i] = t[1][i] = 0.f;
    const int mat = lane >> 3, r = lane & 7;
    const int tok = ((mat >> 1) << 3) + r;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const int col = ks * 16 + ((mat & 1) << 3);
        const uint32_t addr = tile + (col >> 6) * chunk_stride + swz128(tok, col & 63);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(addr, b0, b1, b2, b3);
        if (ks & 1) {
            mma_bf16_16816(t[0], qa[ks], b0, b1);
            mma_bf16_16816(t[1], qa[ks], b2, b3);
        } else {
            mma_bf16_16816(s[0], qa[ks], b0, b1);
            mma_bf16_16816(s[1], qa[ks], b2, b3);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        s[0][i] += t[0][i];
        s[1][i] += t[1][i];
    }
}

// Online softmax update for one block.  `s` holds scores already scaled to base 2
// and set to -inf where masked.  The reference max moves only when a row's block max
// exceeds it by more than kRescaleSlack (log2 units): until then exp2(s - m) <= 2^8, so
// neither the bf16 (or fp16) weights nor the fp32 sums can overflow, and most blocks
// skip the rescale of O entirely.  The weights are rounded to bf16 for the PV MMA and l
// sums exactly those rounded weights (so a one-token context returns V exactly).  The
// FP8 decode form (fp8_block.cuh) and the prefill kernel use the same rule.
constexpr float kRescaleSlack = 8.0f;

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <int D>
__device__ __forceinline__ void softmax_update(RowState<D> &st, float (&s)[2][4], uint32_t (&pa)[4]) {
    float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const bool up0 = mx0 > st.m0 + kRescaleSlack;  // false while mx is -inf
    const bool up1 = mx1 > st.m1 + kRescaleSlack;
    if (__any_sync(0xffffffffu, up0 || up1)) {
        // Rows that move get alpha = 2^(old - new) (0 when old = -inf); the others keep
        // alpha = 1 (their m may still be -inf, and -inf - -inf must not appear).
        const float a0 = up0 ? fast_exp2(st.m0 - mx0) : 1.f;
        const float a1 = up1 ? fast_exp2(st.m1 - mx1) : 1.f;
        if (up0) st.m0 = mx0;
        if (up1) st.m1 = mx1;
        st.l0 *= a0;
        st.l1 *= a1;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            st.o[n][0] *= a0;
            st.o[n][1] *= a0;
            st.o[n][2] *= a1;
            st.o[n][3] *= a1;
        }
    }
    // A row that has seen nothing visible keeps m = -inf: subtract 0 (its weights are 0).
    const float b0 = st.m0 == -INFINITY ? 0.f : st.m0;
    const float b1 = st.m1 == -INFINITY ? 0.f : st.m1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const float e0 = fast_exp2(s[nt][0] - b0), e1 = fast_exp2(s[nt][1] - b0);
        const float e2 = fast_exp2(s[nt][2] - b1), e3 = fast_exp2(s[nt][3] - b1);
        const uint32_t p01 = pack_bf16x2(e0, e1), p23 = pack_bf16x2(e2, e3);
        ps0 += bf16_lo(p01) + bf16_hi(p01);
        ps1 += bf16_lo(p23) + bf16_hi(p23);
        pa[nt * 2 + 0] = p01;
        pa[nt * 2 + 1] = p23;
    }
    st.l0 += ps0;
    st.l1 += ps1;
}

// O += P V for one block; V rows at or past `valid` are zeroed in the fragments (they
// hold whatever the pool held, possibly NaN, and 0 * NaN would poison the sum).
// MASKED = false skips the zeroing when all 16 rows are inside the context.
template <int D, bool MASKED>
__device__ __forceinline__ void pv_block(RowState<D> &st, const uint32_t (&pa)[4], uint32_t tile,
                                         uint32_t chunk_stride, int valid, int lane) {
    const int q4 = lane & 3;
    const int mat = lane >> 3, r = lane & 7;
    const int tok = ((mat & 1) << 3) + r;
    uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
    if (MASKED) {
        keep_lo = (2 * q4 < valid ? 0x0000ffffu : 0u) | (2 * q4 + 1 < valid ? 0xffff0000u : 0u);
        keep_hi = (8 + 2 * q4 < valid ? 0x0000ffffu : 0u) | (8 + 2 * q4 + 1 < valid ? 0xffff0000u : 0u);
    }
#pragma unroll
    for (int n2 = 0; n2 < D / 16; ++n2) {
        const int col = n2 * 16 + ((mat >> 1) << 3);
        const uint32_t addr = tile + (col >> 6) * chunk_stride + swz128(tok, col & 63);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(addr, b0, b1, b2, b3);
        if (MASKED) {
            b0 &= keep_lo;
            b1 &= keep_hi;
            b2 &= keep_lo;
            b3 &= keep_hi;
        }
        mma_bf16_16816(st.o[2 * n2], pa, b0, b1);
        mma_bf16_16816(st.o[2 * n2 + 1], pa, b2, b3);
    }
}

// Reduces l over the quad of lanes that share a row (each lane summed its own columns).
template <int D>
__device__ __forceinline__ void finish_sums(RowState<D> &st) {
    st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, 1);
    st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, 2);
    st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, 1);
    st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, 2);
}

// Programmatic dependent launch: wait for the previous kernel in the stream (and
// everything before it) to finish and publish its memory / let the next kernel start
// its launch.  Both are no-ops when the kernel was launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The dynamic shared memory a kernel has been allowed on each device (one record per
// kernel, kept by its launcher).
struct SmemAllowance {
    std::atomic<int> bytes[64];
};

// Raises `kernel`'s dynamic shared-memory limit to `smem` on the current device unless an
// earlier call already allowed at least that much, so the attribute call leaves the
// per-launch path after a kernel's first launch on a device.
template <typename... Params>
cudaError_t allow_dynamic_smem(void (*kernel)(Params...), size_t smem, SmemAllowance &rec) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (rec.bytes[dev].load(std::memory_order_acquire) >= (int)smem) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int cur = rec.bytes[dev].load(std::memory_order_relaxed);
    while (cur < (int)smem && !rec.bytes[dev].compare_exchange_weak(cur, (int)smem)) {
    }
    return cudaSuccess;
}

// Launches `kernel` on `stream` with programmatic stream serialization, so that its
// launch overlaps the tail of the previous kernel (the kernel calls pdl_wait before it
// touches memory).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace pkv
