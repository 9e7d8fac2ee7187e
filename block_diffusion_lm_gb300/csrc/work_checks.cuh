// Debug-build checks of work-list records (compiled with CSBP_DEBUG_CHECKS).
// With compute-sanitizer unavailable, a kernel built this way validates the
// records its CTA is about to use before any load, store or MMA, and refuses
// the work (DEV_BADWORK in the status word) if one points outside the list or
// names a tile outside the sequence.
#pragma once

#include <cstdint>

#include "csbp_internal.h"

namespace csbp {

// A task record (kTaskWords words) and its segments: the copy index is 0 or
// 1, the tile lies in [0, nT), the segments lie inside the n_segs records and
// each spans a non-empty tile range inside [0, nT), and the task's tile count
// equals their total length.
__device__ __forceinline__ bool task_record_ok(const int32_t* tw, const int32_t* segs, int n_segs,
                                               int nT) {
  const int stream = tw[0], tile = tw[1], sb = tw[3], sc = tw[4], cost = tw[5];
  if (stream < 0 || stream > 1 || tile < 0 || tile >= nT) return false;
  if (sb < 0 || sc < 0 || sb > n_segs - sc) return false;
  int64_t sum = 0;
  for (int k = 0; k < sc; ++k) {
    const int32_t* g = segs + static_cast<int64_t>(sb + k) * kSegWords;
    if (g[0] < 0 || g[0] > 1 || g[1] < 0 || g[1] >= g[2] || g[2] > nT) return false;
    sum += g[2] - g[1];
  }
  return sum == cost;
}

}  // namespace csbp
