// paged_decode.cu -- the decode attention kernel over a block-paged KV cache (sm_103a)
// and its launcher; the CTA body is decode_cta.cuh, the merge of split contexts
// merge.cuh.
#include "decode_cta.cuh"

namespace pkv {

template <int D, bool FP8, int NTH>
__global__ void __launch_bounds__(288, 1)
paged_decode_kernel(const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map, const DecodeArgs a) {
    decode_cta<D, FP8, NTH>(k_map, v_map, a, (int)blockIdx.x, a.grid, true);
}

template __global__ void paged_decode_kernel<64, false, 1>(const __grid_constant__ CUtensorMap,
                                                        const __grid_constant__ CUtensorMap, const DecodeArgs);
template __global__ void paged_decode_kernel<64, false, 2>(const __grid_constant__ CUtensorMap,
                                                        const __grid_constant__ CUtensorMap, const DecodeArgs);
template __global__ void paged_decode_kernel<128, false, 1>(const __grid_constant__ CUtensorMap,
                                                         const __grid_constant__ CUtensorMap, const DecodeArgs);
template __global__ void paged_decode_kernel<128, false, 2>(const __grid_constant__ CUtensorMap,
                                                         const __grid_constant__ CUtensorMap, const DecodeArgs);
template __global__ void paged_decode_kernel<128, true, 1>(const __grid_constant__ CUtensorMap,
                                                           const __grid_constant__ CUtensorMap, const DecodeArgs);
template __global__ void paged_decode_kernel<128, true, 2>(const __grid_constant__ CUtensorMap,
                                                        const __grid_constant__ CUtensorMap, const DecodeArgs);

// ---- host-side launch ----------------------------------------------------------

size_t decode_smem_bytes(int stage_bytes, int num_stages, int num_items) {
    return 1024 + (size_t)num_stages * stage_bytes + 2 * 8 * (size_t)num_stages + 36 * 4 +
           4 * (size_t)(num_items + 1);
}

template <int D, bool FP8, int NTH>
static cudaError_t launch_decode_d(const CUtensorMap &k_map, const CUtensorMap &v_map,
                                   const DecodeArgs &a, size_t smem, cudaStream_t stream) {
    const int ncw = a.heads_per_cta * a.warps_per_head;
    static SmemAllowance allowed;
    cudaError_t e = allow_dynamic_smem(paged_decode_kernel<D, FP8, NTH>, smem, allowed);
    if (e != cudaSuccess) return e;
    e = launch_pdl(paged_decode_kernel<D, FP8, NTH>, dim3(a.grid), dim3((ncw + 1) * 32), smem, stream, k_map,
                   v_map, a);
    if (e != cudaSuccess) return e;
    MergeArgs m;
    m.jobs = a.ws_jobs;
    m.ws_ml = a.ws_ml;
    m.ws_o = a.ws_o;
    m.out = a.out;
    m.slot_rows = a.heads_per_cta * a.group;
    m.num_heads = a.num_heads;
    return launch_merge<D>(m, a.grid, stream);
}

cudaError_t launch_paged_decode(int head_dim, bool fp8, const CUtensorMap &k_map, const CUtensorMap &v_map,
                                const DecodeArgs &a, size_t smem, cudaStream_t stream) {
    if (fp8 && head_dim != 128) return cudaErrorInvalidValue;
    // NTH: n-tiles of 8 query heads per consumer warp
    const bool two = a.group > 8;
    if (fp8) return two ? launch_decode_d<128, true, 2>(k_map, v_map, a, smem, stream)
                        : launch_decode_d<128, true, 1>(k_map, v_map, a, smem, stream);
    if (head_dim == 128)
        return two ? launch_decode_d<128, false, 2>(k_map, v_map, a, smem, stream)
                   : launch_decode_d<128, false, 1>(k_map, v_map, a, smem, stream);
    return two ? launch_decode_d<64, false, 2>(k_map, v_map, a, smem, stream)
               : launch_decode_d<64, false, 1>(k_map, v_map, a, smem, stream);
}

}  // namespace pkv
