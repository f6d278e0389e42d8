// The Markov-clustering step around the expansion C = M * M (Trident page, section 5.7: after
// the SpGEMM, normalize the columns, prune the entries below a threshold, square the remaining
// entries element-wise).  Column sums by fp64 reductions into L2; a row count of the kept
// entries, a device scan into the pruned matrix's row offsets, then a warp-per-row ordered
// compaction (ballot + prefix popcount) that writes (C[i,j] / colsum[j])^2.
#include <algorithm>

#include "internal.h"

namespace sg {

namespace {

__global__ void k_col_sums(const int32_t* __restrict__ col, const double* __restrict__ val, int64_t nnz,
                           double* __restrict__ sums) {
  for (int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; p < nnz;
       p += static_cast<int64_t>(gridDim.x) * blockDim.x)
    atomicAdd(&sums[col[p]], val[p]);
}

__device__ __forceinline__ bool kept(int32_t c, double v, const double* sums, double thr) {
  return v / sums[c] >= thr;
}

// counts[i] = entries of row i whose normalized value is at least thr; one warp per row
__global__ void __launch_bounds__(256) k_keep_count(const int64_t* __restrict__ rp, const int32_t* __restrict__ col,
                                                    const double* __restrict__ val, int64_t rows,
                                                    const double* __restrict__ sums, double thr,
                                                    int64_t* __restrict__ counts) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (row >= rows) return;
  int64_t n = 0;
  for (int64_t p = rp[row] + lane; p < rp[row + 1]; p += 32) n += kept(col[p], val[p], sums, thr) ? 1 : 0;
  for (int d = 16; d > 0; d >>= 1) n += __shfl_xor_sync(0xffffffffu, n, d);
  if (lane == 0) counts[row] = n;
}

// the kept entries of each row, in C's order, at out_rp[row]; one warp per row
__global__ void __launch_bounds__(256) k_keep_write(const int64_t* __restrict__ rp, const int32_t* __restrict__ col,
                                                    const double* __restrict__ val, int64_t rows,
                                                    const double* __restrict__ sums, double thr,
                                                    const int64_t* __restrict__ out_rp, int32_t* __restrict__ out_col,
                                                    double* __restrict__ out_val) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (row >= rows) return;
  int64_t o = out_rp[row];
  const int64_t p1 = rp[row + 1];
  for (int64_t p0 = rp[row]; p0 < p1; p0 += 32) {
    const int64_t p = p0 + lane;
    bool k = false;
    int32_t c = 0;
    double nv = 0.0;
    if (p < p1) {
      c = col[p];
      nv = val[p] / sums[c];
      k = nv >= thr;
    }
    const unsigned b = __ballot_sync(0xffffffffu, k);
    if (k) {
      const int64_t d = o + __popc(b & ((1u << lane) - 1u));
      out_col[d] = c;
      out_val[d] = nv * nv;
    }
    o += __popc(b);
  }
}

}  // namespace

void launch_col_sums(const spgemm_csr& C, double* sums, cudaStream_t s) {
  if (C.nnz == 0) return;
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = std::min<int64_t>(ceil_div(C.nnz, 256), static_cast<int64_t>(sms) * 8);  // grid-stride
  note_launch();
  k_col_sums<<<static_cast<unsigned>(blocks), 256, 0, s>>>(C.col_idx, C.vals, C.nnz, sums);
}

void launch_keep_count(const spgemm_csr& C, const double* sums, double thr, int64_t* counts, cudaStream_t s) {
  if (C.rows == 0) return;
  note_launch();
  k_keep_count<<<static_cast<unsigned>(ceil_div(C.rows, 8)), 256, 0, s>>>(C.row_ptr, C.col_idx, C.vals, C.rows, sums,
                                                                         thr, counts);
}

void launch_keep_write(const spgemm_csr& C, const double* sums, double thr, const int64_t* out_rp, int32_t* out_col,
                       double* out_val, cudaStream_t s) {
  if (C.rows == 0) return;
  note_launch();
  k_keep_write<<<static_cast<unsigned>(ceil_div(C.rows, 8)), 256, 0, s>>>(C.row_ptr, C.col_idx, C.vals, C.rows, sums,
                                                                         thr, out_rp, out_col, out_val);
}

}  // namespace sg
