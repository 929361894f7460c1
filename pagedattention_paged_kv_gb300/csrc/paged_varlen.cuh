// paged_varlen.cuh -- the one-launch varlen step (paged_varlen.cu): decode CTAs and
// chunked-prefill CTAs of one persistent grid, and the cost model that splits the grid.
#pragma once

#include "paged_decode.cuh"
#include "paged_prefill.cuh"

namespace pkv {

// Costs of one unit of each kind of work, from measured rates (see api.cu):
//   dec_sm_us   SM-microseconds a 16-token decode unit costs the CTA that streams it,
//               when few CTAs stream (each at its per-SM rate);
//   dec_gpu_us  microseconds the same unit costs the whole GPU when the decode is bound
//               by HBM bandwidth (the floor on the decode side's time);
//   pre_sm_us   SM-microseconds a prefill unit (16 keys of one tile) costs its CTA.
struct VarlenSplit {
    float dec_sm_us;
    float dec_gpu_us;
    float pre_sm_us;
};

cudaError_t launch_paged_varlen(int head_dim, bool fp8, const CUtensorMap &dk, const CUtensorMap &dv,
                                const DecodeArgs &ad, const CUtensorMap &qm, const CUtensorMap &pk,
                                const CUtensorMap &pv, const PrefillArgs &ap, const PrefillPlan &pp,
                                const VarlenSplit &sp, size_t smem, cudaStream_t stream);

}  // namespace pkv
