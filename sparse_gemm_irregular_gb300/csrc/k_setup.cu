// Setup phase (gMAGNUS page, Algorithm 3, setup part; section III-E binning):
//   * column span of every row of B (for the shortened dense accumulator of narrow rows,
//     gMAGNUS page, section II-B);
//   * per row of A: intermediate products IP[i] = sum over A[i,k] of |B[k,:]| (InterOffsets)
//     and the column span of row i of C, then its bin: heavy (IP > tau), or a light level of
//     the ladder, hash or shortened dense;
//   * a stable multisplit of the rows by bin (count per tile, device scan, scatter), which
//     plays the role of ThreshPartition and of the binning kernel; rows stay in increasing
//     order inside every bin.
#include "internal.h"

namespace sg {

// ---- B row span -----------------------------------------------------------------------
template <int G>
__global__ void k_brow_minmax(const int64_t* __restrict__ rp, const int32_t* __restrict__ col,
                              int64_t rows, int32_t* __restrict__ bmin, int32_t* __restrict__ bmax) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = gid / G;
  const int sub = static_cast<int>(gid % G);
  int32_t lo = 0x7fffffff, hi = -1;
  if (row < rows) {
    for (int64_t p = rp[row] + sub; p < rp[row + 1]; p += G) {
      int32_t c = col[p];
      lo = min(lo, c);
      hi = max(hi, c);
    }
  }
#pragma unroll
  for (int d = G / 2; d > 0; d >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, d));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, d));
  }
  if (row < rows && sub == 0) {
    bmin[row] = lo;
    bmax[row] = hi;
  }
}

static int group_for(int64_t nnz, int64_t rows) {
  int64_t avg = rows > 0 ? nnz / rows : 1;
  if (avg <= 4) return 4;
  if (avg <= 8) return 8;
  if (avg <= 16) return 16;
  return 32;
}

void launch_brow_minmax(const spgemm_csr& B, int32_t* bmin, int32_t* bmax, cudaStream_t s) {
  if (B.rows == 0) return;
  const int g = group_for(B.nnz, B.rows);
  const int64_t threads = B.rows * g;
  const unsigned grid = static_cast<unsigned>(ceil_div(threads, 256));
  switch (g) {
    case 4: note_launch(); k_brow_minmax<4><<<grid, 256, 0, s>>>(B.row_ptr, B.col_idx, B.rows, bmin, bmax); break;
    case 8: note_launch(); k_brow_minmax<8><<<grid, 256, 0, s>>>(B.row_ptr, B.col_idx, B.rows, bmin, bmax); break;
    case 16: note_launch(); k_brow_minmax<16><<<grid, 256, 0, s>>>(B.row_ptr, B.col_idx, B.rows, bmin, bmax); break;
    default: note_launch(); k_brow_minmax<32><<<grid, 256, 0, s>>>(B.row_ptr, B.col_idx, B.rows, bmin, bmax); break;
  }
}

// ---- IP per row, span, bin ---------------------------------------------------------------
__device__ __forceinline__ uint8_t classify_row(int64_t ip, int64_t span, const BinRule& r) {
  if (ip == 0) return kBinEmpty;
  // rows above tau cannot fit a light table: heavy even when all_light is set
  if (ip > r.tau || (r.all_heavy && !r.all_light)) return static_cast<uint8_t>(2 * r.n);
  int L = 0;
  while (L < r.n - 1 && ip > r.upper[L]) ++L;
  const bool dense = !r.no_dense && span <= r.slots[L];
  return static_cast<uint8_t>(2 * L + (dense ? 1 : 0));
}

template <int G>
__global__ void k_row_ip(const int64_t* __restrict__ arp, const int32_t* __restrict__ acol,
                         int64_t rows, const int64_t* __restrict__ brp,
                         const int32_t* __restrict__ bmin, const int32_t* __restrict__ bmax,
                         BinRule rule, int64_t* __restrict__ ip_out, int32_t* __restrict__ lo_out,
                         uint8_t* __restrict__ bin_out) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = gid / G;
  const int sub = static_cast<int>(gid % G);
  int64_t ip = 0;
  int32_t lo = 0x7fffffff, hi = -1;
  if (row < rows) {
    for (int64_t p = arp[row] + sub; p < arp[row + 1]; p += G) {
      const int32_t k = acol[p];
      const int64_t len = brp[k + 1] - brp[k];
      ip += len;
      if (len > 0) {
        lo = min(lo, bmin[k]);
        hi = max(hi, bmax[k]);
      }
    }
  }
#pragma unroll
  for (int d = G / 2; d > 0; d >>= 1) {
    ip += __shfl_xor_sync(0xffffffffu, ip, d);
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, d));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, d));
  }
  if (row < rows && sub == 0) {
    ip_out[row] = ip;
    lo_out[row] = ip > 0 ? lo : 0;
    const int64_t span = ip > 0 ? static_cast<int64_t>(hi) - lo + 1 : 0;
    bin_out[row] = classify_row(ip, span, rule);
  }
}

void launch_row_ip(const spgemm_csr& A, const spgemm_csr& B, const int32_t* bmin,
                   const int32_t* bmax, const BinRule& rule, int64_t* ip, int32_t* span_lo,
                   uint8_t* bin, cudaStream_t s) {
  if (A.rows == 0) return;
  const int g = group_for(A.nnz, A.rows);
  const unsigned grid = static_cast<unsigned>(ceil_div(A.rows * g, 256));
#define SG_ROWIP(G)                                                                            \
  k_row_ip<G><<<grid, 256, 0, s>>>(A.row_ptr, A.col_idx, A.rows, B.row_ptr, bmin, bmax, rule, \
                                   ip, span_lo, bin)
  switch (g) {
    case 4: note_launch(); SG_ROWIP(4); break;
    case 8: note_launch(); SG_ROWIP(8); break;
    case 16: note_launch(); SG_ROWIP(16); break;
    default: note_launch(); SG_ROWIP(32); break;
  }
#undef SG_ROWIP
}

// ---- stable multisplit by bin ------------------------------------------------------------
constexpr int kBinTile = 1024;  // items per block, one per thread
constexpr int kMaxBins = 2 * kMaxLadder + 2;

int64_t bin_blocks(int64_t n) { return ceil_div(n, kBinTile); }

__global__ void __launch_bounds__(kBinTile) k_bin_count(const uint8_t* __restrict__ bin, int64_t n,
                                                        int nbins, int64_t* __restrict__ cnt) {
  __shared__ int c[kMaxBins];
  if (threadIdx.x < kMaxBins) c[threadIdx.x] = 0;
  __syncthreads();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kBinTile + threadIdx.x;
  const int b = i < n ? bin[i] : kBinEmpty;
  const uint32_t peers = __match_any_sync(0xffffffffu, b);  // whole warp, converged
  if (b != kBinEmpty && (peers & lanemask_lt()) == 0) atomicAdd(&c[b], __popc(peers));
  __syncthreads();
  if (threadIdx.x < nbins) cnt[static_cast<int64_t>(threadIdx.x) * gridDim.x + blockIdx.x] = c[threadIdx.x];
}

__global__ void __launch_bounds__(kBinTile) k_bin_scatter(const uint8_t* __restrict__ bin, int64_t n,
                                                          int nbins, const int64_t* __restrict__ off,
                                                          int32_t* __restrict__ out) {
  __shared__ int wc[32][kMaxBins];  // per warp, per bin: count, then exclusive prefix over warps
  const int warp = threadIdx.x >> 5;
  for (int j = threadIdx.x; j < 32 * kMaxBins; j += blockDim.x) (&wc[0][0])[j] = 0;
  __syncthreads();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kBinTile + threadIdx.x;
  const int b = i < n ? bin[i] : kBinEmpty;
  const uint32_t peers = __match_any_sync(0xffffffffu, b);  // whole warp, converged
  if (b != kBinEmpty && (peers & lanemask_lt()) == 0) wc[warp][b] = __popc(peers);
  __syncthreads();
  if (threadIdx.x < nbins) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      int t = wc[w][threadIdx.x];
      wc[w][threadIdx.x] = run;
      run += t;
    }
  }
  __syncthreads();
  if (b != kBinEmpty) {
    const int64_t pos = off[static_cast<int64_t>(b) * gridDim.x + blockIdx.x] + wc[warp][b] +
                        __popc(peers & lanemask_lt());
    out[pos] = static_cast<int32_t>(i);
  }
}

__global__ void k_bin_starts(const int64_t* off, int64_t nblk, int nbins, int64_t* starts) {
  const int b = threadIdx.x;
  if (b <= nbins) starts[b] = off[static_cast<int64_t>(b) * nblk];
}

void launch_bin_count(const uint8_t* bin, int64_t n, int nbins, int64_t* cnt, cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_bin_count<<<static_cast<unsigned>(bin_blocks(n)), kBinTile, 0, s>>>(bin, n, nbins, cnt);
}
void launch_bin_scatter(const uint8_t* bin, int64_t n, int nbins, const int64_t* off, int32_t* out,
                        cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_bin_scatter<<<static_cast<unsigned>(bin_blocks(n)), kBinTile, 0, s>>>(bin, n, nbins, off, out);
}
void launch_bin_starts(const int64_t* off, int64_t nblk, int nbins, int64_t* starts, cudaStream_t s) {
  note_launch();
  k_bin_starts<<<1, 64, 0, s>>>(off, nblk, nbins, starts);
}

// ---- numeric bins of the light hash rows by their exact size -------------------------------
// After the symbolic phase the size of every row of C is known; the numeric hash tables are then
// sized by it (the Ocean page bins the numeric phase by output size), which for power-law rows
// (two to three products per distinct column) shrinks the tables and raises occupancy.
__global__ void k_nnz_bins(const int32_t* __restrict__ rows, int64_t n, const int64_t* __restrict__ rp,
                           BinRule r, uint8_t* __restrict__ bin) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t row = rows[i];
  const int64_t nnz = rp[row + 1] - rp[row];
  int L = 0;
  while (L < r.n - 1 && nnz > r.upper[L]) ++L;
  bin[i] = static_cast<uint8_t>(L);
}
void launch_nnz_bins(const int32_t* rows, int64_t n, const int64_t* row_ptr, const BinRule& rule, uint8_t* bin,
                     cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_nnz_bins<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0, s>>>(rows, n, row_ptr, rule, bin);
}

// ---- optional input validation ------------------------------------------------------------
__global__ void k_validate(const int64_t* __restrict__ rp, const int32_t* __restrict__ col,
                           int64_t rows, int64_t cols, int64_t nnz, uint32_t* err) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < rows) {
    if (rp[i + 1] < rp[i]) set_error(err, kErrCsr);
  }
  if (i == 0 && (rp[0] != 0 || rp[rows] != nnz)) set_error(err, kErrCsr);
  for (int64_t p = i; p < nnz; p += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int32_t c = col[p];
    if (c < 0 || c >= cols) set_error(err, kErrCsr);
  }
}

void launch_validate(const spgemm_csr& M, uint32_t* err, cudaStream_t s) {
  const int64_t work = M.rows > 0 ? M.rows : 1;
  unsigned grid = static_cast<unsigned>(ceil_div(work, 256));
  if (grid > 65535u * 16u) grid = 65535u * 16u;
  note_launch();
  k_validate<<<grid, 256, 0, s>>>(M.row_ptr, M.col_idx, M.rows, M.cols, M.nnz, err);
}

}  // namespace sg
