// Estimation-based row sizing of the light rows (Ocean page: HyperLogLog background, the
// construct-and-merge scheme of Figure 3, Table 1 workflow selection and the overflow
// evaluation).
//
//   * k_hll_sketch: one HyperLogLog sketch of m one-byte registers per row of B.  A column's
//     32-bit hash (the MurmurHash3 finaliser) picks its register by the low log2(m) bits; the
//     register keeps the largest rank (1 + leading zeros of the other 32 - log2(m) bits).
//   * k_hll_rows: the sketch of a row of C is the element-wise maximum of the sketches of the
//     rows of B its row of A selects; the estimate is alpha_m m^2 / sum 2^-register, replaced by
//     linear counting m ln(m / zeros) below 5m/2 (Flajolet et al. 2007, cited by the page), and
//     the capacity is min(IP, ceil(coef * estimate)).  The sum of the 2^-register terms is
//     exact in fp64 in any order (dyadic terms within a 33-bit exponent range), so the result
//     does not depend on the reduction order.
//   * binning by a per-row value, gathers and scatters of per-row offsets, and the copy of the
//     rows from their temporary slots to their final CSR positions (the compaction the
//     estimated workflows need, because C's row sizes are known only after accumulation).
#include <math.h>

#include "internal.h"

namespace sg {

namespace {

__device__ __forceinline__ uint32_t mix32(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85ebca6bu;
  h ^= h >> 13;
  h *= 0xc2b2ae35u;
  h ^= h >> 16;
  return h;
}

// 2^-r exactly, for 0 <= r <= 64
__device__ __forceinline__ double pow2_neg(int r) {
  return __longlong_as_double(static_cast<long long>(1023 - r) << 52);
}

template <int M>
__global__ void __launch_bounds__(256) k_hll_sketch(const int64_t* __restrict__ rp, const int32_t* __restrict__ col,
                                                    int64_t nrows, uint8_t* __restrict__ out) {
  constexpr int kBits = M == 32 ? 5 : 6;
  __shared__ unsigned regs[8][M];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + w;
  if (row >= nrows) return;  // uniform per warp
  for (int j = lane; j < M; j += 32) regs[w][j] = 0u;
  __syncwarp();
  const int64_t b0 = rp[row], b1 = rp[row + 1];
  for (int64_t q = b0 + lane; q < b1; q += 32) {
    const uint32_t h = mix32(static_cast<uint32_t>(col[q]));
    const uint32_t rest = h >> kBits;  // 32 - kBits significant bits
    const unsigned rank = static_cast<unsigned>(__clz(rest)) - kBits + 1u;  // rest == 0: 33 - kBits
    atomicMax(&regs[w][h & (M - 1)], rank);
  }
  __syncwarp();
  for (int j = lane; j < M; j += 32) out[row * M + j] = static_cast<uint8_t>(regs[w][j]);
}

struct HllConst {
  double lc[65];  // lc[v] = m ln(m / v), v = 1..m (host libm)
  double alpha, coef;
};

// One warp per listed row of A (all rows when rows == nullptr).  Writes cap[row] and, if
// requested, est_out[i] (the raw estimate, for the workflow sample).
template <int M>
__global__ void __launch_bounds__(256) k_hll_rows(const int64_t* __restrict__ arp, const int32_t* __restrict__ acol,
                                                  const int32_t* __restrict__ rows, int64_t n,
                                                  const int64_t* __restrict__ ip, const uint8_t* __restrict__ sk,
                                                  HllConst c, int64_t* __restrict__ cap, double* __restrict__ est_out) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * 8 + w;
  if (i >= n) return;
  const int64_t row = rows ? rows[i] : i;
  const int64_t a0 = arp[row], a1 = arp[row + 1];
  unsigned r0 = 0u, r1 = 0u;  // registers 2 lane, 2 lane + 1 (M = 64) or register lane (M = 32)
  constexpr int kU = 4;
  for (int64_t e0 = a0; e0 < a1; e0 += kU) {
    unsigned v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      v[u] = 0u;
      if (e0 + u < a1) {
        const int64_t k = acol[e0 + u];
        if (M == 64) v[u] = reinterpret_cast<const uint16_t*>(sk + k * M)[lane];
        else v[u] = sk[k * M + lane];
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      r0 = max(r0, v[u] & 0xffu);
      if (M == 64) r1 = max(r1, v[u] >> 8);
    }
  }
  double z = pow2_neg(static_cast<int>(r0)) + (M == 64 ? pow2_neg(static_cast<int>(r1)) : 0.0);
  int zeros = (r0 == 0u ? 1 : 0) + (M == 64 && r1 == 0u ? 1 : 0);
  for (int d = 16; d > 0; d >>= 1) {
    z += __shfl_xor_sync(0xffffffffu, z, d);
    zeros += __shfl_xor_sync(0xffffffffu, zeros, d);
  }
  if (lane != 0) return;
  double e = c.alpha * static_cast<double>(M) * static_cast<double>(M) / z;
  if (e <= 2.5 * M && zeros > 0) e = c.lc[zeros];
  if (est_out) est_out[i] = e;
  const int64_t bound = ip[row];
  int64_t k = static_cast<int64_t>(ceil(c.coef * e));
  if (k < 1) k = 1;
  cap[row] = bound > 0 ? (k < bound ? k : bound) : 0;
}

__global__ void k_val_bins(const int32_t* __restrict__ rows, int64_t n, const int64_t* __restrict__ val, BinRule r,
                           uint8_t* __restrict__ bin) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t v = val[rows[i]];
  int L = 0;
  while (L < r.n - 1 && v > r.upper[L]) ++L;
  bin[i] = static_cast<uint8_t>(L);
}

__global__ void k_overflow_bins(const int32_t* __restrict__ rows, int64_t n, const int64_t* __restrict__ est_nnz,
                                const uint8_t* __restrict__ create_bin, int wide_from, uint8_t* __restrict__ bin) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int32_t row = rows[i];
  bin[i] = est_nnz[row] < 0 ? 2 : (create_bin[row] >= wide_from ? 1 : 0);
}

__global__ void k_scatter_off(const int32_t* __restrict__ rows, int64_t n, const int64_t* __restrict__ off,
                              int64_t base, int64_t* __restrict__ dst) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) dst[rows[i]] = base + off[i];
}

// Rows inside [row_begin, row_end) move from their temporary slot to their final position
// (row_ptr[row] - row_ptr[row_begin]), LANES lanes per listed row: 8 for the rows of the warp
// bins (short rows still fill the warp), 32 for the rows of the block bins (long rows).
template <int LANES>
__global__ void __launch_bounds__(256) k_copy_rows(const int32_t* __restrict__ rows, int64_t n,
                                                   const int64_t* __restrict__ row_tmp,
                                                   const int64_t* __restrict__ row_ptr, int64_t row_begin,
                                                   int64_t row_end, const int32_t* __restrict__ tcol,
                                                   const double* __restrict__ tval, int32_t* __restrict__ ccol,
                                                   double* __restrict__ cval) {
  const int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / LANES;
  const int gl = threadIdx.x % LANES;
  if (i >= n) return;
  const int64_t row = rows[i];
  if (row < row_begin || row >= row_end) return;
  const int64_t d = row_ptr[row] - row_ptr[row_begin];
  const int64_t len = row_ptr[row + 1] - row_ptr[row];
  const int64_t src = row_tmp[row];
  for (int64_t j = gl; j < len; j += LANES) {
    ccol[d + j] = tcol[src + j];
    cval[d + j] = tval[src + j];
  }
}

__global__ void k_row_products(const int64_t* __restrict__ arp, const int32_t* __restrict__ acol, int64_t m,
                               const int64_t* __restrict__ brp, int64_t* __restrict__ ip) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= m) return;
  int64_t t = 0;
  for (int64_t e = arp[i]; e < arp[i + 1]; ++e) {
    const int32_t k = acol[e];
    t += brp[k + 1] - brp[k];
  }
  ip[i] = t;
}

}  // namespace

void launch_row_products(const spgemm_csr& A, const spgemm_csr& B, int64_t* ip, cudaStream_t s) {
  if (A.rows == 0) return;
  note_launch();
  k_row_products<<<static_cast<unsigned>(ceil_div(A.rows, 256)), 256, 0, s>>>(A.row_ptr, A.col_idx, A.rows,
                                                                              B.row_ptr, ip);
}

bool hll_registers_ok(int m) { return m == 32 || m == 64; }

void launch_hll_sketch(const spgemm_csr& B, int m, uint8_t* out, cudaStream_t s) {
  if (B.rows == 0) return;
  const unsigned grid = static_cast<unsigned>(ceil_div(B.rows, 8));
  note_launch();
  if (m == 32) k_hll_sketch<32><<<grid, 256, 0, s>>>(B.row_ptr, B.col_idx, B.rows, out);
  else k_hll_sketch<64><<<grid, 256, 0, s>>>(B.row_ptr, B.col_idx, B.rows, out);
}

void launch_hll_rows(const spgemm_csr& A, const int32_t* rows, int64_t n, const int64_t* ip, const uint8_t* sk,
                     int m, double coef, int64_t* cap, double* est_out, cudaStream_t s) {
  if (n == 0) return;
  HllConst c{};
  for (int v = 1; v <= m; ++v) c.lc[v] = m * log(static_cast<double>(m) / v);
  c.alpha = m == 32 ? 0.697 : 0.709;
  c.coef = coef;
  const unsigned grid = static_cast<unsigned>(ceil_div(n, 8));
  note_launch();
  if (m == 32) k_hll_rows<32><<<grid, 256, 0, s>>>(A.row_ptr, A.col_idx, rows, n, ip, sk, c, cap, est_out);
  else k_hll_rows<64><<<grid, 256, 0, s>>>(A.row_ptr, A.col_idx, rows, n, ip, sk, c, cap, est_out);
}

void launch_val_bins(const int32_t* rows, int64_t n, const int64_t* val, const BinRule& rule, uint8_t* bin,
                     cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_val_bins<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0, s>>>(rows, n, val, rule, bin);
}

void launch_overflow_bins(const int32_t* rows, int64_t n, const int64_t* est_nnz, const uint8_t* create_bin,
                          int wide_from, uint8_t* bin, cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_overflow_bins<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0, s>>>(rows, n, est_nnz, create_bin, wide_from,
                                                                          bin);
}

void launch_scatter_off(const int32_t* rows, int64_t n, const int64_t* off, int64_t base, int64_t* dst,
                        cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_scatter_off<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0, s>>>(rows, n, off, base, dst);
}

void launch_copy_rows(const int32_t* rows, int64_t n, const int64_t* row_tmp, const int64_t* row_ptr,
                      int64_t row_begin, int64_t row_end, const int32_t* tcol, const double* tval, int32_t* ccol,
                      double* cval, bool wide, cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  if (wide)
    k_copy_rows<32><<<static_cast<unsigned>(ceil_div(n, 8)), 256, 0, s>>>(rows, n, row_tmp, row_ptr, row_begin,
                                                                          row_end, tcol, tval, ccol, cval);
  else
    k_copy_rows<8><<<static_cast<unsigned>(ceil_div(n, 32)), 256, 0, s>>>(rows, n, row_tmp, row_ptr, row_begin,
                                                                          row_end, tcol, tval, ccol, cval);
}

}  // namespace sg
