// kv_quant.cuh -- the FP8 (e4m3) quantisation of new K/V elements, shared by the KV
// write kernel and the decode kernel's fused KV write.
//
// An element x (bf16) is stored as the e4m3 code nearest to fp32(x) / scale: one IEEE
// round-to-nearest division, then the round-to-nearest-even conversion that saturates
// at +-448 (the largest finite e4m3 value).
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace pkv {

__device__ __forceinline__ uint32_t e4m3_of(uint32_t bf16_bits, float scale) {
    const float y = __fdiv_rn(__uint_as_float(bf16_bits << 16), scale);
    return (uint32_t)__nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3);
}

// Four bf16 (two 32-bit words, low half first) -> four codes in one word, lowest first.
__device__ __forceinline__ uint32_t e4m3x4_of(uint32_t w0, uint32_t w1, float scale) {
    return e4m3_of(w0 & 0xFFFFu, scale) | (e4m3_of(w0 >> 16, scale) << 8) |
           (e4m3_of(w1 & 0xFFFFu, scale) << 16) | (e4m3_of(w1 >> 16, scale) << 24);
}

}  // namespace pkv
