// Expand-sort-compact accumulator for short light rows (Ocean page: ESC accumulators for rows
// with few intermediate products, part of its hybrid accumulator scheme).  One warp per row of
// at most 64 products, all in registers: every lane holds products f = lane and f = lane + 32
// (column as key, A value times B value), a bitonic network sorts the 64 keys across the warp
// with shuffles, equal keys become adjacent and a segmented scan sums each run, and the last
// element of every run is written in column order.  No shared memory, no atomics.
#include <climits>

#include "internal.h"

namespace sg {

namespace {

constexpr int kEscMax = 64;  // products per row

// lane j of the warp holds the inclusive prefix incl of the staged entries' product counts;
// returns the number of entries whose range ends at or before f (the entry holding f)
__device__ __forceinline__ int entry_of(int incl, int f) {
  int pos = 0;
#pragma unroll
  for (int step = 16; step > 0; step >>= 1) {
    const int e = __shfl_sync(0xffffffffu, incl, pos + step - 1);
    if (e <= f) pos += step;
  }
  const int last = __shfl_sync(0xffffffffu, incl, 31);
  if (pos == 31 && last <= f) pos = 32;
  return pos;
}

template <bool NUMERIC>
__global__ void __launch_bounds__(256) k_esc(const int64_t* __restrict__ arp, const int32_t* __restrict__ acol,
                                             const double* __restrict__ aval, const int64_t* __restrict__ brp,
                                             const int32_t* __restrict__ bcol, const double* __restrict__ bval,
                                             const int32_t* __restrict__ rows, int64_t n, Sink sk, uint32_t* err) {
  const int lane = threadIdx.x & 31;
  const int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (i >= n) return;  // uniform per warp
  const int64_t row = rows[i];
  if (NUMERIC && (row < sk.row_begin || row >= sk.row_end)) return;
  int32_t k[2] = {INT_MAX, INT_MAX};
  double v[2] = {0.0, 0.0};
  int base = 0;  // products staged so far
  const int64_t a0 = arp[row], a1 = arp[row + 1];
  for (int64_t e0 = a0; e0 < a1; e0 += 32) {
    const int64_t e = e0 + lane;
    int len = 0;
    int64_t bs = 0;
    double av = 0.0;
    if (e < a1) {
      const int32_t kc = acol[e];
      bs = brp[kc];
      len = static_cast<int>(brp[kc + 1] - bs);
      if (NUMERIC) av = aval[e];
    }
    const int incl = warp_incl_scan(len);
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (base + total > kEscMax) {  // the row is not short: the binning sent it here by mistake
      if (lane == 0) set_error(err, kErrBounds);
      return;
    }
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int f = lane + 32 * s - base;  // this slot's product inside the staged entries
      const int j = entry_of(incl, f < 0 ? 0 : f);
      const int jj = j < 31 ? j : 31;
      const int64_t bj = __shfl_sync(0xffffffffu, bs, jj);
      const int ej = __shfl_sync(0xffffffffu, incl - len, jj);
      const double aj = __shfl_sync(0xffffffffu, av, jj);
      if (f >= 0 && f < total) {
        const int64_t q = bj + (f - ej);
        k[s] = bcol[q];
        if (NUMERIC) v[s] = aj * bval[q];
      }
    }
    base += total;
  }
  // bitonic sort of the 64 keys (element index lane + 32 s), ascending; equal keys stay put
#pragma unroll
  for (int size = 2; size <= kEscMax; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride == 32) {  // elements lane and lane + 32 of the same thread (size 64: ascending)
        if (k[0] > k[1]) {
          const int32_t tk = k[0];
          k[0] = k[1];
          k[1] = tk;
          if (NUMERIC) {
            const double tv = v[0];
            v[0] = v[1];
            v[1] = tv;
          }
        }
      } else {
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          const int el = lane + 32 * s;
          const int32_t ok = __shfl_xor_sync(0xffffffffu, k[s], stride);
          const double ov = NUMERIC ? __shfl_xor_sync(0xffffffffu, v[s], stride) : 0.0;
          const bool up = (el & size) == 0, lower = (el & stride) == 0;
          const bool take = lower == up ? ok < k[s] : ok > k[s];
          if (take) {
            k[s] = ok;
            if (NUMERIC) v[s] = ov;
          }
        }
      }
    }
  }
  // run boundaries: element e is the last of its run when e = 63 or key[e + 1] differs (every
  // shuffle runs on all lanes; the selects come after)
  const int32_t dn0 = __shfl_down_sync(0xffffffffu, k[0], 1);
  const int32_t first1 = __shfl_sync(0xffffffffu, k[1], 0);
  const int32_t dn1 = __shfl_down_sync(0xffffffffu, k[1], 1);
  const int32_t next0 = lane < 31 ? dn0 : first1;
  const bool tail0 = k[0] != INT_MAX && next0 != k[0];
  const bool tail1 = k[1] != INT_MAX && (lane == 31 || dn1 != k[1]);
  const unsigned b0 = __ballot_sync(0xffffffffu, tail0), b1 = __ballot_sync(0xffffffffu, tail1);
  const int count = __popc(b0) + __popc(b1);
  if (!NUMERIC) {
    if (lane == 0) sk.row_nnz[row] = count;
    return;
  }
  // segmented inclusive sums (a run starts where the previous key differs)
  const int32_t prev0 = __shfl_up_sync(0xffffffffu, k[0], 1);
  const int32_t pv1 = __shfl_up_sync(0xffffffffu, k[1], 1);
  const int32_t last0 = __shfl_sync(0xffffffffu, k[0], 31);
  const int32_t prev1 = lane > 0 ? pv1 : last0;
  bool h0 = lane == 0 || prev0 != k[0];
  bool h1 = prev1 != k[1];
  double x0 = v[0], x1 = v[1];
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const double y0 = __shfl_up_sync(0xffffffffu, x0, d), y1 = __shfl_up_sync(0xffffffffu, x1, d);
    const bool g0 = __shfl_up_sync(0xffffffffu, h0, d), g1 = __shfl_up_sync(0xffffffffu, h1, d);
    if (lane >= d) {
      if (!h0) x0 += y0;
      if (!h1) x1 += y1;
      h0 = h0 || g0;
      h1 = h1 || g1;
    }
  }
  // the run that crosses from element 31 to element 32 carries the first half's partial sum
  const double carry = __shfl_sync(0xffffffffu, x0, 31);
  if (!h1) x1 += carry;  // no run start between element 32 and this one
  const int64_t rp0 = sk.row_ptr[row];
  const int64_t expected = sk.row_ptr[row + 1] - rp0;
  if (count != expected) {
    if (lane == 0) set_error(err, kErrRowOverflow);
    return;
  }
  const int64_t out = rp0 - sk.row_ptr[sk.row_begin];
  const unsigned lt = (1u << lane) - 1u;
  if (tail0) {
    const int64_t d = out + __popc(b0 & lt);
    sk.c_col[d] = k[0];
    sk.c_val[d] = x0;
  }
  if (tail1) {
    const int64_t d = out + __popc(b0) + __popc(b1 & lt);
    sk.c_col[d] = k[1];
    sk.c_val[d] = x1;
  }
}

}  // namespace

int64_t esc_max_products() { return kEscMax; }

void launch_esc(const spgemm_csr& A, const spgemm_csr& B, const int32_t* rows, int64_t n, bool numeric,
                const Sink& sink, uint32_t* err, cudaStream_t s) {
  if (n == 0) return;
  const unsigned grid = static_cast<unsigned>(ceil_div(n, 8));
  note_launch();
  if (numeric)
    k_esc<true><<<grid, 256, 0, s>>>(A.row_ptr, A.col_idx, A.vals, B.row_ptr, B.col_idx, B.vals, rows, n, sink, err);
  else
    k_esc<false><<<grid, 256, 0, s>>>(A.row_ptr, A.col_idx, A.vals, B.row_ptr, B.col_idx, B.vals, rows, n, sink, err);
}

}  // namespace sg
