// attn_block.cuh -- pieces shared by the decode and the chunked-prefill kernels: the
// online softmax's rescale rule, fp16 packing, programmatic dependent launch and the
// per-kernel shared-memory allowance.
#pragma once

#include <atomic>

#include <cuda_fp16.h>

#include "pkv_common.cuh"

namespace pkv {

// The online softmax's lazy rescale: a row's reference max moves only when its block max
// exceeds it by more than kRescaleSlack (log2 units); until then exp2(s - m) <= 2^8, so
// neither the 16-bit weights nor the fp32 sums can overflow, and most blocks skip the
// rescale of O entirely.  The decode forms (bf16t_block.cuh, fp8_block.cuh) and the
// prefill CTAs use the same rule.
constexpr float kRescaleSlack = 8.0f;

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
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
