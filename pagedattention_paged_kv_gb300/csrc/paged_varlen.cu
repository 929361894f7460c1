// paged_varlen.cu -- one launch for a whole continuous-batching iteration: the decode rows
// and the prefill chunks of a varlen batch run side by side in one persistent grid.
//
// Method: "Servis Motor İçleri: PagedAttention, Sürekli Batching, parçalanmış Prefill"
// (aiengineeringfromscratch.com, Phase 17 - 04), "What the scheduler looks like": every
// iteration runs one fused forward over a batch that mixes single-token decodes with
// ~512-token prompt chunks ("Chunked prefill protects the TTFT tail").
//
// GB300 design
//  * The two kinds of work want different parts of the chip: a decode is bound by HBM
//    (every cached byte is read once), a chunk by the tensor cores.  Run one after the
//    other, each leaves the other's resource idle, and the iteration costs their sum.
//  * Every CTA first counts both kinds of work (16-token decode units, 16-key prefill
//    units) and then takes a role: CTAs [0, k) run the decode body (decode_cta.cuh) over
//    the decode units, CTAs [k, grid) the chunked-prefill body (prefill_cta.cuh) over
//    the prefill units, each side with its own balanced split and merge jobs.  k is the
//    same in every CTA: it minimises the larger of the two sides' modelled times, a decode
//    unit costing a CTA its bytes at the per-SM streaming rate (never faster than the
//    whole HBM allows) and a prefill unit its FLOPs at the per-SM tensor rate
//    (VarlenSplit, measured rates passed by the host).  Compressed onto a few SMs the
//    decode streams at its per-SM limit instead of waiting on HBM on every SM, which
//    frees SM time for the chunk.
//  * The two merges (decode parts, prefill parts) follow as their own launches.
#include "decode_cta.cuh"
#include "prefill_cta.cuh"
#include "paged_varlen.cuh"

namespace pkv {

// Decode CTAs out of G (1 <= k <= G - 1): one CTA of each role always runs, because each
// side's CTA 0 writes that side's merge jobs and the zero rows of its empty items.
__device__ __forceinline__ int decode_ctas(int64_t Td, int64_t Tp, int G, const VarlenSplit &sp) {
    if (Td == 0) return 1;
    if (Tp == 0) return G - 1;
    const float d_sm = (float)Td * sp.dec_sm_us, d_hbm = (float)Td * sp.dec_gpu_us;
    const float p_sm = (float)Tp * sp.pre_sm_us;
    int best = 1;
    float best_t = INFINITY;
    for (int k = 1; k < G; ++k) {
        const float t = fmaxf(fmaxf(d_sm / (float)k, d_hbm), p_sm / (float)(G - k));
        if (t < best_t) {
            best_t = t;
            best = k;
        }
    }
    return best;
}

// Sum over the CTA of one value per thread (all threads call it); `red` holds 32 int64.
__device__ __forceinline__ int64_t cta_sum(int64_t x, int64_t *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) red[warp] = x;
    __syncthreads();
    int64_t t = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
    __syncthreads();
    return t;
}

template <int D, bool FP8>
__global__ void __launch_bounds__(kPrefillThreads, 1)
paged_varlen_kernel(const __grid_constant__ CUtensorMap dk_map, const __grid_constant__ CUtensorMap dv_map,
                    const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap pk_map,
                    const __grid_constant__ CUtensorMap pv_map, const DecodeArgs ad, const PrefillArgs ap,
                    const VarlenSplit sp) {
    extern __shared__ uint8_t smem_raw[];
    int64_t *red = reinterpret_cast<int64_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    pdl_wait();
    pdl_trigger();
    // Work of each kind (no error reporting here: each side's CTA 0 reports its own).
    int64_t td = 0, tp = 0;
    const int V = ad.num_seqs * ad.head_tiles;
    for (int v = threadIdx.x; v < V; v += blockDim.x) td += item_blocks(ad, v, false);
    for (int s = threadIdx.x; s < ap.num_seqs; s += blockDim.x) tp += seq_units(ap, s, false);
    td = cta_sum(td, red);
    tp = cta_sum(tp, red);  // ends with __syncthreads: the bodies may now reuse the memory
    const int G = (int)gridDim.x;
    const int k = decode_ctas(td, tp, G, sp);
    if ((int)blockIdx.x < k) decode_cta<D, FP8, 1>(dk_map, dv_map, ad, (int)blockIdx.x, k, false);
    else prefill_cta<D, FP8>(q_map, pk_map, pv_map, ap, (int)blockIdx.x - k, G - k, false);
}

template <int D, bool FP8>
static cudaError_t launch_varlen_d(const CUtensorMap &dk, const CUtensorMap &dv, const DecodeArgs &ad,
                                   const CUtensorMap &qm, const CUtensorMap &pk, const CUtensorMap &pv,
                                   const PrefillArgs &ap, const PrefillPlan &pp, const VarlenSplit &sp,
                                   size_t smem, cudaStream_t stream) {
    static_assert(!FP8 || D == 128, "the FP8 cache path is built for head_dim 128");
    auto kernel = paged_varlen_kernel<D, FP8>;
    static SmemAllowance allowed;
    cudaError_t e = allow_dynamic_smem(kernel, smem, allowed);
    if (e != cudaSuccess) return e;
    if (ad.grid != ap.grid) return cudaErrorInvalidValue;
    e = launch_pdl(kernel, dim3(ap.grid), dim3(kPrefillThreads), smem, stream, dk, dv, qm, pk, pv, ad, ap, sp);
    if (e != cudaSuccess) return e;
    MergeArgs m;
    m.jobs = ad.ws_jobs;
    m.ws_ml = ad.ws_ml;
    m.ws_o = ad.ws_o;
    m.out = ad.out;
    m.slot_rows = ad.heads_per_cta * ad.group;
    m.num_heads = ad.num_heads;
    e = launch_merge<D>(m, ad.grid, stream);
    if (e != cudaSuccess) return e;
    m.jobs = ap.ws_jobs;
    m.ws_ml = ap.ws_ml;
    m.ws_o = ap.ws_o;
    m.out = ap.out;
    m.slot_rows = pp.rows;
    m.num_heads = ap.num_heads;
    return launch_merge<D>(m, ap.grid, stream);
}

cudaError_t launch_paged_varlen(int head_dim, bool fp8, const CUtensorMap &dk, const CUtensorMap &dv,
                                const DecodeArgs &ad, const CUtensorMap &qm, const CUtensorMap &pk,
                                const CUtensorMap &pv, const PrefillArgs &ap, const PrefillPlan &pp,
                                const VarlenSplit &sp, size_t smem, cudaStream_t stream) {
    if (fp8) {
        if (head_dim != 128) return cudaErrorInvalidValue;
        return launch_varlen_d<128, true>(dk, dv, ad, qm, pk, pv, ap, pp, sp, smem, stream);
    }
    return head_dim == 128 ? launch_varlen_d<128, false>(dk, dv, ad, qm, pk, pv, ap, pp, sp, smem, stream)
                           : launch_varlen_d<64, false>(dk, dv, ad, qm, pk, pv, ap, pp, sp, smem, stream);
}

}  // namespace pkv
