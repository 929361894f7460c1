// reshape_and_cache.cu -- the KV write (sm_103a).
//
// "vLLM推理引擎架构PagedAttention机制与高吞吐推理" (lpnh.cn) §2.2: the pool is
// [num_blocks, block_size, num_kv_heads, head_dim] for K and for V, so slot
// (block * block_size + offset) of the pool starts num_kv_heads * head_dim elements
// times the slot into the array.  Each new token's K row and V row are copied there
// unchanged (bit-exact).
//
// One warp per (token, K-or-V) row: the row (num_kv_heads * head_dim * 2 bytes,
// 2 KiB for Llama-70B shapes) moves as 16-byte vectors, fully coalesced on both sides.
// The source is read once (no L1 allocation); the destination is written normally.
#include "attn_block.cuh"
#include "kv_quant.cuh"
#include "pkv_common.cuh"

namespace pkv {

__global__ void __launch_bounds__(256)
reshape_and_cache_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                         const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                         const int64_t *__restrict__ slot_mapping, int64_t num_tokens,
                         int64_t num_slots, int row_vecs, int *err) {
    pdl_wait();  // the rows and slots may come from the previous kernel in the stream
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
         w < 2 * num_tokens; w += warps) {
        const int64_t t = w >> 1;
        const bool is_v = (w & 1) != 0;
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;  // padding token
        if (slot >= num_slots) {
            if (lane == 0 && !is_v) flag_error(err, PKV_DEVERR_SLOT);
            continue;
        }
        const uint4 *src = (is_v ? v : k) + t * row_vecs;
        uint4 *dst = (is_v ? v_cache : k_cache) + slot * row_vecs;
        for (int i = lane; i < row_vecs; i += 32) dst[i] = __ldcs(src + i);
    }
}

// FP8 cache: one warp per (token, K-or-V) row; a lane turns 16 bf16 (32 bytes, two
// 16-byte loads) into 16 codes (one 16-byte store) with e4m3x4_of (kv_quant.cuh).

__global__ void __launch_bounds__(256)
reshape_and_cache_fp8_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                             const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                             const int64_t *__restrict__ slot_mapping, int64_t num_tokens,
                             int64_t num_slots, int row_groups, float k_scale, float v_scale,
                             int *err) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
         w < 2 * num_tokens; w += warps) {
        const int64_t t = w >> 1;
        const bool is_v = (w & 1) != 0;
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;  // padding token
        if (slot >= num_slots) {
            if (lane == 0 && !is_v) flag_error(err, PKV_DEVERR_SLOT);
            continue;
        }
        const float sc = is_v ? v_scale : k_scale;
        const uint4 *src = (is_v ? v : k) + t * row_groups * 2;  // 16 bf16 = 2 vectors
        uint4 *dst = (is_v ? v_cache : k_cache) + slot * row_groups;  // 16 codes = 1 vector
        for (int i = lane; i < row_groups; i += 32) {
            const uint4 a = __ldcs(src + 2 * i), b = __ldcs(src + 2 * i + 1);
            dst[i] = make_uint4(e4m3x4_of(a.x, a.y, sc), e4m3x4_of(a.z, a.w, sc), e4m3x4_of(b.x, b.y, sc),
                                e4m3x4_of(b.z, b.w, sc));
        }
    }
}

cudaError_t launch_reshape_and_cache_fp8(void *k_cache, void *v_cache, const void *k, const void *v,
                                         const int64_t *slot_mapping, int64_t num_tokens,
                                         int64_t num_slots, int row_elems, float k_scale,
                                         float v_scale, int num_sms, int *err, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int warps_per_cta = 8;
    int64_t ctas = (2 * num_tokens + warps_per_cta - 1) / warps_per_cta;
    const int64_t cap = (int64_t)num_sms * 8;
    if (ctas > cap) ctas = cap;
    return launch_pdl(reshape_and_cache_fp8_kernel, dim3((unsigned)ctas), dim3(warps_per_cta * 32), 0,
                      stream, static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache),
                      static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping,
                      num_tokens, num_slots, row_elems / 16, k_scale, v_scale, err);
}

// Copy-on-write support: for each (src, dst) pair, block dst of both caches becomes a
// copy of block src.  One CTA per pair (grid-stride), 16-byte vectors.
__global__ void __launch_bounds__(256)
copy_blocks_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                   const int32_t *__restrict__ pairs, int64_t num_pairs, int64_t num_blocks,
                   int64_t block_vecs, int *err) {
    pdl_wait();
    pdl_trigger();
    for (int64_t p = blockIdx.x; p < num_pairs; p += gridDim.x) {
        const int32_t src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (threadIdx.x == 0) flag_error(err, PKV_DEVERR_BLOCK_ID);
            continue;
        }
        const uint4 *ks = k_cache + src * block_vecs, *vs = v_cache + src * block_vecs;
        uint4 *kd = k_cache + dst * block_vecs, *vd = v_cache + dst * block_vecs;
        for (int64_t i = threadIdx.x; i < block_vecs; i += blockDim.x) {
            kd[i] = ks[i];
            vd[i] = vs[i];
        }
    }
}

cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, const int32_t *pairs, int64_t num_pairs,
                               int64_t num_blocks, int64_t block_bytes, int num_sms, int *err,
                               cudaStream_t stream) {
    if (num_pairs == 0) return cudaSuccess;
    int64_t ctas = num_pairs;
    if (ctas > (int64_t)num_sms * 4) ctas = (int64_t)num_sms * 4;
    return launch_pdl(copy_blocks_kernel, dim3((unsigned)ctas), dim3(256), 0, stream,
                      static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), pairs, num_pairs,
                      num_blocks, block_bytes / 16, err);
}

cudaError_t launch_reshape_and_cache(void *k_cache, void *v_cache, const void *k, const void *v,
                                     const int64_t *slot_mapping, int64_t num_tokens,
                                     int64_t num_slots, int row_bytes, int num_sms, int *err,
                                     cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int warps_per_cta = 8;
    int64_t ctas = (2 * num_tokens + warps_per_cta - 1) / warps_per_cta;
    const int64_t cap = (int64_t)num_sms * 8;
    if (ctas > cap) ctas = cap;
    return launch_pdl(reshape_and_cache_kernel, dim3((unsigned)ctas), dim3(warps_per_cta * 32), 0,
                      stream, static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache),
                      static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping,
                      num_tokens, num_slots, row_bytes / 16, err);
}

}  // namespace pkv
