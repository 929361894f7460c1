// pkv_split.cuh -- how a persistent grid shares a flat list of work units.
//
// T units (16-token KV blocks of all work items laid end to end) are cut into
// `ge` contiguous shares of equal size (+-1): CTA c takes [c*T/ge, (c+1)*T/ge).
// A share can begin or end inside an item; such partial results go to workspace
// slot 2c (the CTA's first item) or 2c+1 (its last item), and a merge kernel adds
// them up.  Only a CTA's first and last items can be partial, so 2 * grid slots
// always suffice whatever the batch.
#pragma once

#include <stdint.h>

namespace pkv {

// CTAs that take part: all of `grid`, unless that would leave fewer than
// `min_units` units per CTA.
__device__ __forceinline__ int split_ctas(int64_t T, int grid, int min_units) {
    if (T <= 0) return 1;
    int64_t g = T / min_units;
    if (g < 1) g = 1;
    if (g > grid) g = grid;
    return (int)g;
}

__device__ __forceinline__ int64_t share_begin(int c, int64_t T, int ge) {
    return (int64_t)c * T / ge;
}

// The CTA whose share holds unit f (0 <= f < T).
__device__ __forceinline__ int share_owner(int64_t f, int64_t T, int ge) {
    return (int)(((f + 1) * ge + T - 1) / T - 1);
}

// Workspace slot of CTA c's part of the item that begins at unit item_begin.
__device__ __forceinline__ int part_slot(int c, int64_t item_begin, int64_t T, int ge) {
    return item_begin <= share_begin(c, T, ge) ? 2 * c : 2 * c + 1;
}

}  // namespace pkv
