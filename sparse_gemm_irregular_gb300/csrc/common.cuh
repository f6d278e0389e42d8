// Shared device and host helpers of the SpGEMM library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/spgemm.h"

namespace sg {

constexpr int32_t kEmptyKey = -1;          // empty hash slot (columns are >= 0)
constexpr int32_t kPadKey = 0x7fffffff;    // sorts after every column

// Bits of the device error word (set by kernels, read by the host at sync points).
enum DevErr : uint32_t {
  kErrHashFull = 1u,       // a hash probe sequence exceeded the table
  kErrBounds = 2u,         // an index left its range (inconsistent input or a planner bug)
  kErrRowOverflow = 4u,    // a row wrote more entries than the symbolic phase counted
  kErrCsr = 8u,            // input validation failed
  kErrTimeout = 16u,       // a bounded wait on an asynchronous copy gave up
};

__device__ __forceinline__ void set_error(uint32_t* err, uint32_t bit) { atomicOr(err, bit); }

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }
__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Multiplicative hash of a column (Knuth's golden-ratio constant), reduced to [0, slots)
// with a high multiply, so any table size works ("modulo hashing", gMAGNUS page, III-E).
__device__ __forceinline__ uint32_t hash_slot(int32_t col, uint32_t slots) {
  return __umulhi(static_cast<uint32_t>(col) * 2654435761u, slots);
}

template <typename T>
__device__ __forceinline__ T warp_incl_scan(T v) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    T o = __shfl_up_sync(0xffffffffu, v, d);
    if (static_cast<int>(lane_id()) >= d) v += o;
  }
  return v;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// Block-wide inclusive scan.  `tmp` holds at least 33 T in shared memory.  Every thread of
// the block must call it.  Returns the inclusive prefix; *total receives the block sum.
template <typename T>
__device__ __forceinline__ T block_incl_scan(T v, T* tmp, T* total) {
  const int warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  T x = warp_incl_scan(v);
  if (lane_id() == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    T w = (static_cast<int>(lane_id()) < nw) ? tmp[lane_id()] : T(0);
    w = warp_incl_scan(w);
    if (static_cast<int>(lane_id()) < nw) tmp[lane_id()] = w;
    if (lane_id() == 31) tmp[32] = w;
  }
  __syncthreads();
  if (warp > 0) x += tmp[warp - 1];
  if (total) *total = tmp[32];
  __syncthreads();
  return x;
}

// Largest index i in [lo, hi) with a[i] <= key (a non-decreasing, a[lo] <= key assumed).
template <typename T>
__device__ __forceinline__ int64_t upper_bound_minus1(const T* a, int64_t lo, int64_t hi, T key) {
  while (hi - lo > 1) {
    int64_t mid = lo + ((hi - lo) >> 1);
    if (a[mid] <= key) lo = mid; else hi = mid;
  }
  return lo;
}

__host__ __device__ constexpr int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

__host__ __device__ inline int ilog2_i64(int64_t x) {  // floor(log2(x)), x >= 1
  int r = 0;
  while (x > 1) { x >>= 1; ++r; }
  return r;
}

}  // namespace sg
