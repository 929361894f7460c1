// transfer.cu -- a step's host <-> device transfers done by the SMs (sm_103a).
//
// On a GB300 the GPU reaches page-locked host memory through its NVLink-C2C port, so a
// kernel can load (or store) host memory directly.  For the few MB a decode step moves
// (queries and new K/V rows in, outputs back) the copy engines run at ~120-130 GB/s and
// take ~20 us each way; many SM threads with independent 16-byte accesses in flight move
// the same bytes in a few microseconds.  The kernel is an ordinary copy: src and dst are
// device-accessible addresses (one of them a mapped page-locked host buffer), `bytes`
// bytes, any alignment (the 16-byte body goes as vectors when both sides allow it).
#include "pkv_common.cuh"
#include "attn_block.cuh"

namespace pkv {

// VPT independent 16-byte vectors per thread per pass, all loads before any store.
constexpr int kCopyVecPerThread = 4;

__global__ void __launch_bounds__(256)
copy_vec_kernel(uint4 *__restrict__ dst, const uint4 *__restrict__ src, int64_t n16) {
    pdl_wait();  // the source may come from the previous kernel in the stream
    pdl_trigger();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x * kCopyVecPerThread;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x * kCopyVecPerThread + threadIdx.x; base < n16;
         base += stride) {
        uint4 v[kCopyVecPerThread];
#pragma unroll
        for (int k = 0; k < kCopyVecPerThread; ++k) {
            const int64_t i = base + (int64_t)k * blockDim.x;
            if (i < n16) v[k] = __ldcs(src + i);
        }
#pragma unroll
        for (int k = 0; k < kCopyVecPerThread; ++k) {
            const int64_t i = base + (int64_t)k * blockDim.x;
            if (i < n16) __stcs(dst + i, v[k]);
        }
    }
}

__global__ void __launch_bounds__(256)
copy_bytes_kernel(uint8_t *__restrict__ dst, const uint8_t *__restrict__ src, int64_t n) {
    pdl_wait();
    pdl_trigger();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

cudaError_t launch_copy(void *dst, const void *src, int64_t bytes, int num_sms, cudaStream_t stream) {
    if (bytes <= 0) return cudaSuccess;
    const uintptr_t d = reinterpret_cast<uintptr_t>(dst), s = reinterpret_cast<uintptr_t>(src);
    if (((d | s) & 15) == 0) {
        const int64_t n16 = bytes / 16, tail = bytes - n16 * 16;
        if (n16 > 0) {
            const int64_t per_cta = 256LL * kCopyVecPerThread;
            int64_t ctas = (n16 + per_cta - 1) / per_cta;
            if (ctas > (int64_t)num_sms * 8) ctas = (int64_t)num_sms * 8;
            cudaError_t e = launch_pdl(copy_vec_kernel, dim3((unsigned)ctas), dim3(256), 0, stream,
                                       static_cast<uint4 *>(dst), static_cast<const uint4 *>(src), n16);
            if (e != cudaSuccess) return e;
        }
        if (tail == 0) return cudaSuccess;
        return launch_pdl(copy_bytes_kernel, dim3(1), dim3(256), 0, stream, static_cast<uint8_t *>(dst) + n16 * 16,
                          static_cast<const uint8_t *>(src) + n16 * 16, tail);
    }
    int64_t ctas = (bytes + 255) / 256;
    if (ctas > (int64_t)num_sms * 8) ctas = (int64_t)num_sms * 8;
    return launch_pdl(copy_bytes_kernel, dim3((unsigned)ctas), dim3(256), 0, stream, static_cast<uint8_t *>(dst),
                      static_cast<const uint8_t *>(src), bytes);
}

}  // namespace pkv
