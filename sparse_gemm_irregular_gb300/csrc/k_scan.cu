// Device-wide exclusive prefix sum of int64 values (reduce, scan of tile sums, scan + add).
// Used for C.row_ptr (gMAGNUS page, Algorithm 3, PrefixSum), the C^ row pointers, the slice
// offsets of the outer product and every bin / chunk offset array.  Three passes over the
// data, no inter-block waiting.
#include "internal.h"

namespace sg {

constexpr int kScanThreads = 512;
constexpr int kScanItems = kScanTile / kScanThreads;  // 8

__global__ void __launch_bounds__(kScanThreads) k_tile_sums(const int64_t* __restrict__ in,
                                                             int64_t n, int64_t* __restrict__ sums) {
  __shared__ int64_t tmp[33];
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kScanTile;
  int64_t s = 0;
#pragma unroll
  for (int j = 0; j < kScanItems; ++j) {
    int64_t i = base + j * kScanThreads + threadIdx.x;
    if (i < n) s += in[i];
  }
  s = warp_sum(s);
  if (lane_id() == 0) tmp[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    int64_t v = threadIdx.x < kScanThreads / 32 ? tmp[threadIdx.x] : 0;
    v = warp_sum(v);
    if (threadIdx.x == 0) sums[blockIdx.x] = v;
  }
}

// Scan one tile (each thread owns kScanItems consecutive elements) and add `carry[blockIdx]`.
__global__ void __launch_bounds__(kScanThreads) k_tile_scan(const int64_t* in, int64_t* out,
                                                             int64_t n, const int64_t* carry,
                                                             int64_t* total_out) {
  __shared__ int64_t tmp[33];
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kScanTile + threadIdx.x * kScanItems;
  int64_t v[kScanItems];
  int64_t local = 0;
#pragma unroll
  for (int j = 0; j < kScanItems; ++j) {
    v[j] = (base + j < n) ? in[base + j] : 0;
    local += v[j];
  }
  int64_t tot;
  int64_t incl = block_incl_scan(local, tmp, &tot);
  int64_t run = incl - local + (carry ? carry[blockIdx.x] : 0);
#pragma unroll
  for (int j = 0; j < kScanItems; ++j) {
    if (base + j < n) out[base + j] = run;
    run += v[j];
  }
  if (total_out && blockIdx.x == gridDim.x - 1 && threadIdx.x == blockDim.x - 1) *total_out = run;
}

int64_t scan_scratch_elems(int64_t n) {
  int64_t need = 0;
  while (n > kScanTile) {
    n = ceil_div(n, kScanTile);
    need += n + 1;
  }
  return need + 1;
}

void scan_excl_i64(const int64_t* in, int64_t* out, int64_t n, int64_t* scratch, cudaStream_t s) {
  if (n <= 0) {
    cudaMemsetAsync(out, 0, sizeof(int64_t), s);
    return;
  }
  const int64_t nb = ceil_div(n, kScanTile);
  if (nb == 1) {
    note_launch();
    k_tile_scan<<<1, kScanThreads, 0, s>>>(in, out, n, nullptr, out + n);
    return;
  }
  int64_t* sums = scratch;  // nb + 1
  note_launch();
  k_tile_sums<<<static_cast<unsigned>(nb), kScanThreads, 0, s>>>(in, n, sums);
  scan_excl_i64(sums, sums, nb, scratch + nb + 1, s);  // sums[nb] = total
  note_launch();
  k_tile_scan<<<static_cast<unsigned>(nb), kScanThreads, 0, s>>>(in, out, n, sums, nullptr);
  cudaMemcpyAsync(out + n, sums + nb, sizeof(int64_t), cudaMemcpyDeviceToDevice, s);
}

}  // namespace sg
