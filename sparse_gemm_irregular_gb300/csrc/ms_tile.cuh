// Tile helpers shared by the histogram and multisplit kernels (gMAGNUS page, section III-C,
// Algorithm 5).  Every kernel uses the same static partition: tile t holds elements
// [t*kMsTile, (t+1)*kMsTile) of C^, each thread kMsItems consecutive ones, and the rows of C^
// the tile touches (at most group_rows when every row holds more than tau elements; processed
// in windows of group_rows rows otherwise).
#pragma once

#include "internal.h"

namespace sg {

constexpr int kMsItems = static_cast<int>(kMsTile) / kMsThreads;  // 8 per thread
static_assert(kMsItems * kMsThreads == kMsTile && kMsItems % 4 == 0, "tile shape");

template <bool VALS>
__device__ __forceinline__ void ms_load_tile(const int32_t* __restrict__ col, const double* __restrict__ val,
                                             int64_t p0, int64_t g1, int32_t (&c)[kMsItems],
                                             double (&v)[kMsItems]) {
  if (p0 + kMsItems <= g1) {
#pragma unroll
    for (int j = 0; j < kMsItems; j += 4) {
      const int4 x = __ldcs(reinterpret_cast<const int4*>(col + p0 + j));
      c[j] = x.x; c[j + 1] = x.y; c[j + 2] = x.z; c[j + 3] = x.w;
    }
    if (VALS) {
#pragma unroll
      for (int j = 0; j < kMsItems; j += 2) {
        const double2 d = __ldcs(reinterpret_cast<const double2*>(val + p0 + j));
        v[j] = d.x;
        v[j + 1] = d.y;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < kMsItems; ++j) {
      c[j] = (p0 + j < g1) ? col[p0 + j] : 0;
      if (VALS) v[j] = (p0 + j < g1) ? val[p0 + j] : 0.0;
    }
  }
}

// Bins (local row * v + chunk) of a thread's 8 consecutive elements inside row window
// [rstart[0], rstart[nr]); -1 outside the tile or the window.
__device__ __forceinline__ void ms_bins(const int64_t* rstart, int nr, int64_t p0, int64_t g1,
                                        const int32_t (&c)[kMsItems], int shift, int64_t v, int (&bin)[kMsItems],
                                        uint32_t* err) {
  int r = 0;
  while (r + 1 < nr && p0 >= rstart[r + 1]) ++r;
#pragma unroll
  for (int j = 0; j < kMsItems; ++j) {
    const int64_t p = p0 + j;
    while (r + 1 < nr && p >= rstart[r + 1]) ++r;
    int b = -1;
    if (p < g1 && p >= rstart[0] && p < rstart[nr]) {
      const int64_t ch = static_cast<int64_t>(c[j]) >> shift;
      if (c[j] >= 0 && ch < v) b = static_cast<int>(r * v + ch);
      else set_error(err, kErrBounds);
    }
    bin[j] = b;
  }
}

template <bool MATCH>
__device__ __forceinline__ void ms_count(unsigned* hist, int b) {
  if (MATCH) {
    // warp-aggregated: one shared-memory atomic per distinct bin per warp
    const uint32_t peers = __match_any_sync(0xffffffffu, b);
    if (b >= 0 && (peers & lanemask_lt()) == 0) atomicAdd(&hist[b], __popc(peers));
  } else if (b >= 0) {
    atomicAdd(&hist[b], 1u);
  }
}

template <bool MATCH>
__device__ __forceinline__ unsigned ms_rank(unsigned* hist, int b) {
  // count and rank in one step: the group's atomic returns the bin's count so far
  if (MATCH) {
    const uint32_t peers = __match_any_sync(0xffffffffu, b);
    const int leader = __ffs(peers) - 1;
    unsigned base = 0;
    if (b >= 0 && static_cast<int>(lane_id()) == leader) base = atomicAdd(&hist[b], __popc(peers));
    base = __shfl_sync(0xffffffffu, base, leader);
    return base + __popc(peers & lanemask_lt());
  }
  return b >= 0 ? atomicAdd(&hist[b], 1u) : 0u;
}

}  // namespace sg
