// Heavy rows (gMAGNUS page, sections III-A to III-C, Algorithms 3-5):
//   MaskedCsr2Csc   -> csc_count / csc_scatter: A[x_heavy,:] transposed by a counting sort.
//   sliceOffsets    -> slice_sizes + scan: |column k of A~_CSC| * |row k of B|.
//   OuterProduct    -> outer_product: flattened static partition of all slice elements,
//                      one atomic reservation per (A~ entry, block) on the C^ row cursor,
//                      coalesced copy of (partial) B rows scaled by the A value.
//   Histogram       -> histogram: per (C^ row, chunk) counts, warp-aggregated with
//                      __match_any_sync into a block histogram, one global atomic per bin.
//   ThreshPartition -> chunk_partition + the stable bin scatter: heavy chunks first.
//   Multisplit      -> multisplit: block histogram whose warp-aggregated atomics also rank every
//                      element inside its bin, one global reservation per bin, then every
//                      element is written at (its bin's reserved run + its rank) with the
//                      column shifted into the chunk's local range.
// plus the bookkeeping that turns the final chunks into offsets inside the rows of C.
#include <algorithm>

#include "internal.h"
#include "ms_tile.cuh"

namespace sg {

// ---- small helpers --------------------------------------------------------------------------
__global__ void k_gather_ip(const int32_t* __restrict__ rows, int64_t n, const int64_t* __restrict__ ip,
                            int64_t* __restrict__ out) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) out[i] = ip[rows[i]];
}
void launch_gather_ip(const int32_t* heavy_rows, int64_t nrows, const int64_t* ip, int64_t* out,
                      cudaStream_t s) {
  if (nrows == 0) return;
  note_launch();
  k_gather_ip<<<static_cast<unsigned>(ceil_div(nrows, 256)), 256, 0, s>>>(heavy_rows, nrows, ip, out);
}

__global__ void k_copy_i64(const int64_t* __restrict__ a, int64_t* __restrict__ b, int64_t n) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) b[i] = a[i];
}
void launch_copy_i64(const int64_t* src, int64_t* dst, int64_t n, cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_copy_i64<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0, s>>>(src, dst, n);
}

__global__ void k_offset_copy(const int64_t* __restrict__ a, int64_t n, int64_t delta, int64_t* __restrict__ b) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) b[i] = a[i] - delta;
}
void launch_offset_copy(const int64_t* src, int64_t n, int64_t delta, int64_t* dst, cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_offset_copy<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0, s>>>(src, n, delta, dst);
}

__global__ void k_list_sums(const int32_t* __restrict__ list, int64_t n, const int64_t* __restrict__ a,
                            const int64_t* __restrict__ b, unsigned long long* out) {
  unsigned long long sa = 0, sb = 0;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    sa += static_cast<unsigned long long>(a[list[i]]);
    sb += static_cast<unsigned long long>(b[list[i]]);
  }
  sa = warp_sum(sa);
  sb = warp_sum(sb);
  if (lane_id() == 0) {
    atomicAdd(&out[0], sa);
    atomicAdd(&out[1], sb);
  }
}
void launch_list_sums(const int32_t* list, int64_t n, const int64_t* a, const int64_t* b, unsigned long long* out,
                      cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_list_sums<<<static_cast<unsigned>(std::min<int64_t>(ceil_div(n, 256), 1024)), 256, 0, s>>>(list, n, a, b, out);
}

// out[i] = src[out[i]]: turn positions of a concatenated list into its elements, in place.
__global__ void k_gather_rows(const int32_t* __restrict__ src, int32_t* __restrict__ io, int64_t n) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) io[i] = src[io[i]];
}
void launch_gather_rows(const int32_t* src, int32_t* io, int64_t n, cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_gather_rows<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0, s>>>(src, io, n);
}

// ---- masked CSR -> CSC of the heavy rows of A ------------------------------------------------
__global__ void k_csc_count(const int64_t* __restrict__ arp, const int32_t* __restrict__ acol,
                            const int32_t* __restrict__ rows, int64_t nrows, int32_t* __restrict__ cnt) {
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (w >= nrows) return;
  const int64_t r = rows[w];
  for (int64_t e = arp[r] + lane_id(); e < arp[r + 1]; e += 32) atomicAdd(&cnt[acol[e]], 1);
}
void launch_csc_count(const spgemm_csr& A, const int32_t* heavy_rows, int64_t nrows, int32_t* colcnt,
                      cudaStream_t s) {
  if (nrows == 0) return;
  note_launch();
  k_csc_count<<<static_cast<unsigned>(ceil_div(nrows * 32, 256)), 256, 0, s>>>(A.row_ptr, A.col_idx,
                                                                               heavy_rows, nrows, colcnt);
}

__global__ void k_slice_sizes(const int32_t* __restrict__ cnt, const int64_t* __restrict__ brp,
                              int64_t kcols, int64_t* __restrict__ colsz, int64_t* __restrict__ slsz) {
  const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (k < kcols) {
    const int64_t c = cnt[k];
    colsz[k] = c;
    slsz[k] = c * (brp[k + 1] - brp[k]);
  }
}
void launch_slice_sizes(const int32_t* colcnt, const spgemm_csr& B, int64_t kcols, int64_t* colptr_sizes,
                        int64_t* slice_sizes, cudaStream_t s) {
  if (kcols == 0) return;
  note_launch();
  k_slice_sizes<<<static_cast<unsigned>(ceil_div(kcols, 256)), 256, 0, s>>>(colcnt, B.row_ptr, kcols,
                                                                            colptr_sizes, slice_sizes);
}

__global__ void k_csc_scatter(const int64_t* __restrict__ arp, const int32_t* __restrict__ acol,
                              const double* __restrict__ aval, const int32_t* __restrict__ rows,
                              int64_t nrows, unsigned long long* __restrict__ cursor,
                              int32_t* __restrict__ crow, double* __restrict__ cval, int32_t* __restrict__ ccol) {
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (w >= nrows) return;
  const int64_t r = rows[w];
  for (int64_t e = arp[r] + lane_id(); e < arp[r + 1]; e += 32) {
    const int32_t k = acol[e];
    const unsigned long long pos = atomicAdd(&cursor[k], 1ull);
    crow[pos] = static_cast<int32_t>(w);  // batch-local heavy row (x_map)
    cval[pos] = aval[e];
    ccol[pos] = k;                        // its column: the slice of the outer product
  }
}
void launch_csc_scatter(const spgemm_csr& A, const int32_t* heavy_rows, int64_t nrows, int64_t* cursor,
                        int32_t* csc_row, double* csc_val, int32_t* csc_col, cudaStream_t s) {
  if (nrows == 0) return;
  note_launch();
  k_csc_scatter<<<static_cast<unsigned>(ceil_div(nrows * 32, 256)), 256, 0, s>>>(
      A.row_ptr, A.col_idx, A.vals, heavy_rows, nrows, reinterpret_cast<unsigned long long*>(cursor),
      csc_row, csc_val, csc_col);
}

// Slice (column of A~_CSC) of entry a of a block whose entries lie in slices [s0, s1]: the column
// recorded by the scatter, checked against the block's range (a binary search over colptr would
// be a chain of dependent loads at the start of every block).
__device__ __forceinline__ int64_t entry_slice(const int32_t* __restrict__ ccol, const int64_t* __restrict__ colptr,
                                               int64_t s0, int64_t s1, int64_t a, uint32_t* err) {
  if (s0 == s1) return s0;
  const int64_t s = ccol[a];
  if (s < s0 || s > s1 || a < colptr[s] || a >= colptr[s + 1]) {
    set_error(err, kErrBounds);
    return upper_bound_minus1(colptr, s0, s1 + 1, a);
  }
  return s;
}

// ---- static partition of a flattened index space (GroupRange + Search, Algorithms 4 and 5) -----
// For every block b covering [b*tile, min(total, (b+1)*tile)): the index of the segment (row of
// C^, or slice of the outer product) holding its first and its last element, found by one
// thread per block boundary in parallel, so no block starts with a serial search.
__global__ void k_partition(const int64_t* __restrict__ off, int64_t nseg, int64_t total, int64_t tile,
                            int64_t nblk, int2* __restrict__ part) {
  const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (b >= nblk) return;
  const int64_t g0 = b * tile;
  const int64_t g1 = min(total, g0 + tile);
  const int64_t s0 = upper_bound_minus1(off, 0, nseg + 1, g0);
  const int64_t s1 = upper_bound_minus1(off, s0, nseg + 1, g1 - 1);
  part[b] = make_int2(static_cast<int>(s0), static_cast<int>(s1));
}
void launch_partition(const int64_t* off, int64_t nseg, int64_t total, int64_t tile, int2* part, cudaStream_t s) {
  const int64_t nblk = ceil_div(total, tile);
  if (nblk == 0) return;
  note_launch();
  k_partition<<<static_cast<unsigned>(ceil_div(nblk, 256)), 256, 0, s>>>(off, nseg, total, tile, nblk, part);
}

// ---- outer product (Algorithm 4) ---------------------------------------------------------------
struct OpSmem {
  int64_t a_first, nent;
};

// With `counts` set, the kernel also produces the level-0 histogram of C^ (elements per
// (row, chunk), chunk = column >> shift): lanes of a warp that write the same (entry, chunk)
// combine their counts with __match_any_sync and the leader adds them to the global counter,
// which saves a separate pass over the columns of C^.
template <bool VALS, bool HIST>
__global__ void __launch_bounds__(kOpThreads) k_outer_product(
    const int64_t* __restrict__ colptr, const int32_t* __restrict__ crow, const double* __restrict__ cval,
    const int32_t* __restrict__ ccol, const int64_t* __restrict__ slice_off, const int2* __restrict__ part,
    int64_t total,
    const int64_t* __restrict__ brp, const int32_t* __restrict__ bcol, const double* __restrict__ bval,
    unsigned long long* __restrict__ cursor, int32_t* __restrict__ out_col, double* __restrict__ out_val,
    unsigned long long* __restrict__ counts, int shift, int64_t v, uint32_t* err) {
  extern __shared__ __align__(16) char smem_raw[];
  __shared__ OpSmem hdr;
  int64_t* dst_delta = reinterpret_cast<int64_t*>(smem_raw);
  int64_t* src_delta = dst_delta + kOpTile;
  int32_t* seg_start = reinterpret_cast<int32_t*>(src_delta + kOpTile);

  const int64_t g0 = static_cast<int64_t>(blockIdx.x) * kOpTile;
  const int64_t g1 = min(total, g0 + kOpTile);
  const int2 sp = part[blockIdx.x];
  const int64_t s0 = sp.x, s1 = sp.y;
  if (threadIdx.x == 0) {
    // ARange (GetAEntry, Eq. 3): first and last entry of A~_CSC touched by this block
    const int64_t len0 = brp[s0 + 1] - brp[s0];
    const int64_t len1 = brp[s1 + 1] - brp[s1];
    const int64_t a_first = colptr[s0] + (g0 - slice_off[s0]) / len0;
    const int64_t a_last = colptr[s1] + (g1 - 1 - slice_off[s1]) / len1;
    hdr.a_first = a_first;
    hdr.nent = a_last - a_first + 1;
  }
  __syncthreads();
  const int64_t a_first = hdr.a_first, nent = hdr.nent;
  if (nent > kOpTile || nent <= 0) {  // impossible for consistent offsets
    if (threadIdx.x == 0) set_error(err, kErrBounds);
    return;
  }
  // Step 2: reserve space in the C^ rows, one atomic per (entry, block) (GetExcess trims the
  // partial B rows at both ends of the block's range).
  for (int64_t e = threadIdx.x; e < nent; e += blockDim.x) {
    const int64_t a = a_first + e;
    const int64_t s = entry_slice(ccol, colptr, s0, s1, a, err);
    const int64_t b0 = brp[s];
    const int64_t len = brp[s + 1] - b0;
    const int64_t F = slice_off[s] + (a - colptr[s]) * len;
    const int64_t lo = max(F, g0), hi = min(F + len, g1);
    const int64_t cnt = hi > lo ? hi - lo : 0;
    const int64_t clo = lo < g1 ? lo : g1;
    int64_t base = 0;
    if (cnt > 0) base = static_cast<int64_t>(atomicAdd(&cursor[crow[a]], static_cast<unsigned long long>(cnt)));
    seg_start[e] = static_cast<int32_t>(clo - g0);
    dst_delta[e] = base - (clo - g0);
    src_delta[e] = b0 + (clo - F) - (clo - g0);
  }
  __syncthreads();
  // Step 3: populate C^, consecutive threads -> consecutive elements of a B row
  const int32_t n = static_cast<int32_t>(g1 - g0);
  int32_t p = threadIdx.x;
  int32_t e = 0;
  if (p < n) {
    int32_t lo = 0, hi = static_cast<int32_t>(nent) - 1;
    while (lo < hi) {  // last entry with seg_start <= p
      const int32_t mid = (lo + hi + 1) >> 1;
      if (seg_start[mid] <= p) lo = mid; else hi = mid - 1;
    }
    e = lo;
  }
  if (!HIST) {
    // kOpUnroll elements per thread per step: all their gathers are issued before the stores
    constexpr int kOpUnroll = 4;
    for (; p < n; p += kOpUnroll * blockDim.x) {
      int64_t dst[kOpUnroll];
      int32_t c[kOpUnroll];
      double a[kOpUnroll], b[kOpUnroll];
#pragma unroll
      for (int u = 0; u < kOpUnroll; ++u) {
        const int32_t q = p + u * static_cast<int32_t>(blockDim.x);
        dst[u] = -1;
        if (q < n) {
          while (e + 1 < nent && seg_start[e + 1] <= q) ++e;
          const int64_t src = src_delta[e] + q;
          dst[u] = dst_delta[e] + q;
          c[u] = bcol[src];
          if (VALS) {
            a[u] = __ldg(&cval[a_first + e]);
            b[u] = bval[src];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kOpUnroll; ++u) {
        if (dst[u] < 0) continue;
        out_col[dst[u]] = c[u];
        if (VALS) out_val[dst[u]] = a[u] * b[u];
      }
    }
    return;
  }
  // uniform trip count across the block so that every lane can join the warp match
  for (int32_t p0 = 0; p0 < n; p0 += blockDim.x) {
    p = p0 + static_cast<int32_t>(threadIdx.x);
    int key = -1;
    int64_t row = 0;
    if (p < n) {
      while (e + 1 < nent && seg_start[e + 1] <= p) ++e;
      const int64_t src = src_delta[e] + p;
      const int64_t dst = dst_delta[e] + p;
      const int32_t c = bcol[src];
      out_col[dst] = c;
      if (VALS) out_val[dst] = __ldg(&cval[a_first + e]) * bval[src];
      const int64_t ch = static_cast<int64_t>(c) >> shift;
      row = crow[a_first + e];
      if (c >= 0 && ch < v) key = static_cast<int>(e * v + ch);
      else set_error(err, kErrBounds);
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && (peers & lanemask_lt()) == 0)
      atomicAdd(&counts[row * v + (key & (v - 1))], static_cast<unsigned long long>(__popc(peers)));
  }
}

void launch_outer_product(const int64_t* colptr, const int32_t* csc_row, const double* csc_val,
                          const int32_t* csc_col, const int64_t* slice_off, const int2* part, int64_t total,
                         const spgemm_csr& B,
                          int64_t* row_cursor, int32_t* chat_col, double* chat_val, bool with_vals,
                          unsigned long long* counts, int shift, int64_t nchunks, uint32_t* err, cudaStream_t s) {
  if (total == 0) return;
  const size_t smem = kOpTile * (8 + 8 + 4);
  const unsigned grid = static_cast<unsigned>(ceil_div(total, kOpTile));
  auto* ull = reinterpret_cast<unsigned long long*>(row_cursor);
#define SG_OP(V, H)                                                                                          \
  do {                                                                                                      \
    cudaFuncSetAttribute(k_outer_product<V, H>, cudaFuncAttributeMaxDynamicSharedMemorySize,              \
                         static_cast<int>(smem));                                                           \
    note_launch();                                                                                          \
    k_outer_product<V, H><<<grid, kOpThreads, smem, s>>>(colptr, csc_row, csc_val, csc_col, slice_off, part, \
                                                         total,                                             \
                                                         B.row_ptr, B.col_idx, B.vals, ull, chat_col,        \
                                                         V ? chat_val : nullptr, counts, shift, nchunks, err); \
  } while (0)
  if (with_vals) {
    if (counts) SG_OP(true, true); else SG_OP(true, false);
  } else {
    if (counts) SG_OP(false, true); else SG_OP(false, false);
  }
#undef SG_OP
}

// ---- direct split of level 0 (optional path, SPGEMM_FLAG_DIRECT_SPLIT) ---------------------------
// Chunk histogram of the rows of B: bh[k * v + c] = entries of row k in chunk c (column >> shift).
// Only rows used by heavy A entries (colcnt[k] > 0) are counted.
__global__ void k_b_chunk_hist(const int64_t* __restrict__ brp, const int32_t* __restrict__ bcol, int64_t krows,
                               const int32_t* __restrict__ colcnt, int shift, int64_t v, int32_t* __restrict__ bh,
                               uint32_t* err) {
  const int64_t k = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (k >= krows || colcnt[k] == 0) return;
  for (int64_t q = brp[k] + lane_id(); q < brp[k + 1]; q += 32) {
    const int64_t c = static_cast<int64_t>(bcol[q]) >> shift;
    if (c >= 0 && c < v) atomicAdd(&bh[k * v + c], 1);
    else set_error(err, kErrBounds);
  }
}
void launch_b_chunk_hist(const spgemm_csr& B, const int32_t* colcnt, int shift, int64_t v, int32_t* bh, uint32_t* err,
                         cudaStream_t s) {
  if (B.rows == 0) return;
  note_launch();
  k_b_chunk_hist<<<static_cast<unsigned>(ceil_div(B.rows * 32, 256)), 256, 0, s>>>(B.row_ptr, B.col_idx, B.rows,
                                                                                   colcnt, shift, v, bh, err);
}

// counts[r * v + c] = sum over the entries A[row r, k] of bh[k * v + c]: the level-0 histogram of
// C^ without forming C^ (every product of A[r, k] with row k of B lands in the chunks that row k
// of B touches) -- a sparse (heavy rows of A) times dense (k x v) product.  The entries of the
// heavy rows, in row order (prefix hrp), are split evenly over warps, so the longest rows of a
// power-law A do not serialise on one warp.  Lane c of a warp sums chunk c (chunks in groups of
// 32) while the row stays the same and adds the partial sum to the counter when it changes.
__global__ void k_heavy_row_len(const int64_t* __restrict__ arp, const int32_t* __restrict__ rows, int64_t nrows,
                                int64_t* __restrict__ len) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r < nrows) len[r] = arp[rows[r] + 1] - arp[rows[r]];
}

constexpr int64_t kCountRun = 256;  // entries per warp

__global__ void k_row_chunk_counts(const int64_t* __restrict__ arp, const int32_t* __restrict__ acol,
                                   const int32_t* __restrict__ rows, int64_t nrows, const int64_t* __restrict__ hrp,
                                   const int32_t* __restrict__ bh, int64_t v, unsigned long long* __restrict__ counts) {
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t total = hrp[nrows];
  const int64_t x0 = w * kCountRun;
  if (x0 >= total) return;
  const int64_t x1 = min(total, x0 + kCountRun);
  const int64_t r0 = upper_bound_minus1(hrp, int64_t(0), nrows + 1, x0);  // row holding entry x0
  for (int64_t c0 = 0; c0 < v; c0 += 32) {
    const int64_t c = c0 + lane_id();
    int64_t r = r0;
    int64_t e = arp[rows[r]] + (x0 - hrp[r]);
    unsigned long long sum = 0;
    for (int64_t x = x0; x < x1; ++x, ++e) {
      while (x >= hrp[r + 1]) {  // row change: flush the partial sum of row r
        if (sum && c < v) atomicAdd(&counts[r * v + c], sum);
        sum = 0;
        ++r;
        e = arp[rows[r]];
      }
      if (c < v) sum += static_cast<unsigned long long>(__ldg(&bh[static_cast<int64_t>(__ldg(&acol[e])) * v + c]));
    }
    if (sum && c < v) atomicAdd(&counts[r * v + c], sum);
  }
}
void launch_row_chunk_counts(const spgemm_csr& A, const int32_t* rows, int64_t nrows, const int64_t* hrp,
                             int64_t entries, const int32_t* bh, int64_t v, unsigned long long* counts,
                             cudaStream_t s) {
  if (nrows == 0 || entries == 0) return;
  note_launch();
  const int64_t warps = ceil_div(entries, kCountRun);
  k_row_chunk_counts<<<static_cast<unsigned>(ceil_div(warps * 32, 256)), 256, 0, s>>>(A.row_ptr, A.col_idx, rows,
                                                                                      nrows, hrp, bh, v, counts);
}
void launch_heavy_row_len(const spgemm_csr& A, const int32_t* rows, int64_t nrows, int64_t* len, cudaStream_t s) {
  if (nrows == 0) return;
  note_launch();
  k_heavy_row_len<<<static_cast<unsigned>(ceil_div(nrows, 256)), 256, 0, s>>>(A.row_ptr, rows, nrows, len);
}

// Outer product writing straight into C^_reord: the static partition of Algorithm 4 (tiles of
// kOdTile products over the slices of A~_CSC x B), but each run of consecutive elements that
// belong to one (entry, chunk) reserves its space with one atomic on that C^_reord row's cursor
// (warp runs found with __match_any_sync) and is written with the column shifted into the
// chunk's range.  A tile's first entry and entry count come from the partition kernel (GetAEntry,
// Eq. 3, with its divisions), so a block starts without a serial chain; its entries are staged
// in shared memory kOdWin at a time (position of their first product in the tile, source offset
// in B, row, A value), so any number of entries fits and the shared footprint stays small enough
// for a full SM of blocks.
__global__ void k_od_partition(const int64_t* __restrict__ slice_off, int64_t nseg, int64_t total,
                               const int64_t* __restrict__ colptr, const int64_t* __restrict__ brp, int64_t ntiles,
                               OdTile* __restrict__ tiles) {
  const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (b >= ntiles) return;
  const int64_t g0 = b * kOdTile;
  const int64_t g1 = min(total, g0 + kOdTile);
  // last slice starting at or before the tile's ends: never an empty slice (an empty slice
  // shares its offset with the next one)
  const int64_t s0 = upper_bound_minus1(slice_off, 0, nseg + 1, g0);
  const int64_t s1 = upper_bound_minus1(slice_off, s0, nseg + 1, g1 - 1);
  const int64_t len0 = brp[s0 + 1] - brp[s0];
  const int64_t len1 = brp[s1 + 1] - brp[s1];
  OdTile t;
  t.s0 = static_cast<int32_t>(s0);
  t.s1 = static_cast<int32_t>(s1);
  if (len0 <= 0 || len1 <= 0) {  // inconsistent offsets
    t.a_first = 0;
    t.nent = 0;
  } else {
    t.a_first = colptr[s0] + (g0 - slice_off[s0]) / len0;
    t.nent = colptr[s1] + (g1 - 1 - slice_off[s1]) / len1 - t.a_first + 1;
  }
  tiles[b] = t;
}

void launch_od_partition(const int64_t* slice_off, int64_t nseg, int64_t total, const int64_t* colptr,
                         const spgemm_csr& B, OdTile* tiles, cudaStream_t s) {
  const int64_t ntiles = ceil_div(total, kOdTile);
  if (ntiles == 0) return;
  note_launch();
  k_od_partition<<<static_cast<unsigned>(ceil_div(ntiles, 256)), 256, 0, s>>>(slice_off, nseg, total, colptr,
                                                                              B.row_ptr, ntiles, tiles);
}

template <bool VALS>
__global__ void __launch_bounds__(kOpThreads) k_outer_direct(
    const int64_t* __restrict__ colptr, const int32_t* __restrict__ crow, const double* __restrict__ cval,
    const int32_t* __restrict__ ccol, const int64_t* __restrict__ slice_off, const OdTile* __restrict__ tiles,
    int64_t total, const int64_t* __restrict__ brp, const int32_t* __restrict__ bcol,
    const double* __restrict__ bval, unsigned long long* __restrict__ cursor, int32_t* __restrict__ out_col,
    double* __restrict__ out_val, int shift, int64_t v, uint32_t* err) {
  // per staged entry: where its products start in the tile, B's columns and values of its products
  // indexed by the tile position, its C^_reord row's cursors, and its A value
  __shared__ int32_t seg_start[kOdWin + 1];
  __shared__ const int32_t* seg_bc[kOdWin];
  __shared__ const double* seg_bv[kOdWin];
  __shared__ unsigned long long* seg_cur[kOdWin];
  __shared__ double seg_a[kOdWin];
  const int64_t g0 = static_cast<int64_t>(blockIdx.x) * kOdTile;
  const int64_t g1 = min(total, g0 + kOdTile);
  const OdTile tl = tiles[blockIdx.x];
  const int64_t s0 = tl.s0, s1 = tl.s1, a_first = tl.a_first, nent = tl.nent;
  if (nent <= 0) {
    if (threadIdx.x == 0) set_error(err, kErrBounds);
    return;
  }
  const int32_t n = static_cast<int32_t>(g1 - g0);
  const uint32_t wmask = (1u << shift) - 1u;
  const uint32_t uv = static_cast<uint32_t>(v);
  const int32_t tid = static_cast<int32_t>(threadIdx.x);
  for (int64_t w0 = 0; w0 < nent; w0 += kOdWin) {
    const int32_t wn = static_cast<int32_t>(min(static_cast<int64_t>(kOdWin), nent - w0));
    // the window's entries, and one more: the start of the next window (or the tile's end)
    for (int32_t j = tid; j <= wn; j += static_cast<int32_t>(blockDim.x)) {
      const int64_t e = w0 + j;
      if (e < nent) {
        const int64_t a = a_first + e;
        const int64_t sl = entry_slice(ccol, colptr, s0, s1, a, err);
        const int64_t b0 = brp[sl];
        const int64_t len = brp[sl + 1] - b0;
        const int64_t F = slice_off[sl] + (a - colptr[sl]) * len;
        const int64_t lo = max(F, g0);
        const int64_t clo = lo < g1 ? lo : g1;
        seg_start[j] = static_cast<int32_t>(clo - g0);
        if (j < wn) {
          const int64_t sd = b0 + (clo - F) - (clo - g0);  // B position of tile position 0
          seg_bc[j] = bcol + sd;
          seg_bv[j] = VALS ? bval + sd : nullptr;
          seg_cur[j] = cursor + static_cast<int64_t>(crow[a]) * v;
          seg_a[j] = VALS ? cval[a] : 0.0;
        }
      } else {
        seg_start[j] = n;
      }
    }
    __syncthreads();
    const int32_t plo = seg_start[0], phi = seg_start[wn];
    // this thread's first product: last entry of the window starting at or before it
    int32_t e = 0;
    {
      const int32_t p = plo + tid;
      int32_t lo = 0, hi = wn - 1;
      while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (seg_start[mid] <= p) lo = mid; else hi = mid - 1;
      }
      e = lo;
    }
    for (int32_t p0 = plo; p0 < phi; p0 += static_cast<int32_t>(blockDim.x)) {
      const int32_t p = p0 + tid;
      int key = -1;
      int32_t c = 0;
      double val = 0.0;
      unsigned long long* cur = nullptr;
      if (p < phi) {
        while (e + 1 < wn && seg_start[e + 1] <= p) ++e;
        c = seg_bc[e][p];
        if (VALS) val = seg_a[e] * seg_bv[e][p];
        const uint32_t ch = static_cast<uint32_t>(c) >> shift;  // a negative column lands above v
        if (ch < uv) {
          key = e * static_cast<int>(uv) + static_cast<int>(ch);  // window-local entry: unique in the round
          cur = seg_cur[e] + ch;
        } else {
          set_error(err, kErrBounds);
        }
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, key);
      const int leader = __ffs(peers) - 1;
      unsigned long long base = 0;
      if (key >= 0 && static_cast<int>(lane_id()) == leader)
        base = atomicAdd(cur, static_cast<unsigned long long>(__popc(peers)));
      base = __shfl_sync(0xffffffffu, base, leader);
      if (key >= 0) {
        const int64_t dst = static_cast<int64_t>(base) + __popc(peers & lanemask_lt());
        // evict-first: C^_reord is read back only by the next kernel, while the rows of B the
        // tile reads are reused by the tiles after it
        __stcs(out_col + dst, static_cast<int32_t>(static_cast<uint32_t>(c) & wmask));
        if (VALS) __stcs(out_val + dst, val);
      }
    }
    __syncthreads();
  }
}

void launch_outer_direct(const int64_t* colptr, const int32_t* csc_row, const double* csc_val,
                         const int32_t* csc_col, const int64_t* slice_off, const OdTile* tiles, int64_t total,
                         const spgemm_csr& B, unsigned long long* cursor, int32_t* out_col, double* out_val,
                         bool with_vals, int shift, int64_t nchunks, uint32_t* err, cudaStream_t s) {
  if (total == 0) return;
  const unsigned grid = static_cast<unsigned>(ceil_div(total, kOdTile));
  note_launch();
  if (with_vals)
    k_outer_direct<true><<<grid, kOpThreads, 0, s>>>(colptr, csc_row, csc_val, csc_col, slice_off, tiles, total,
                                                     B.row_ptr, B.col_idx, B.vals, cursor, out_col, out_val, shift,
                                                     nchunks, err);
  else
    k_outer_direct<false><<<grid, kOpThreads, 0, s>>>(colptr, csc_row, csc_val, csc_col, slice_off, tiles, total,
                                                      B.row_ptr, B.col_idx, B.vals, cursor, out_col, nullptr, shift,
                                                      nchunks, err);
}

// ---- histogram and multisplit (Algorithm 5) -----------------------------------------------------
// Tile helpers (static partition, per-thread bins, count and rank): ms_tile.cuh.

template <bool MATCH>
__global__ void __launch_bounds__(kMsThreads) k_histogram(const int64_t* __restrict__ rp, const int2* __restrict__ part,
                                                         int64_t total, int64_t ntiles, const int32_t* __restrict__ col,
                                                         int shift, int64_t v, int64_t gr,
                                                         unsigned long long* __restrict__ counts, uint32_t* err) {
  extern __shared__ __align__(16) char smem_raw[];
  int64_t* rstart = reinterpret_cast<int64_t*>(smem_raw);         // gr + 1
  unsigned* hist = reinterpret_cast<unsigned*>(rstart + gr + 1);  // gr * v
  // persistent blocks: tile t, then t + gridDim.x, ...; the next tile is loaded while the
  // current one is counted
  int64_t t = blockIdx.x;
  if (t >= ntiles) return;
  int32_t c[kMsItems], cn[kMsItems];
  double unused[kMsItems];
  ms_load_tile<false>(col, nullptr, t * kMsTile + static_cast<int64_t>(threadIdx.x) * kMsItems,
                      min(total, (t + 1) * kMsTile), c, unused);
  int2 pr = part[t];
  // row bounds of the first row window, kept in a register by the first gr+1 threads
  int64_t rb = threadIdx.x <= min(gr, static_cast<int64_t>(pr.y - pr.x + 1)) ? rp[pr.x + threadIdx.x] : 0;
  for (; t < ntiles; t += gridDim.x) {
    const int64_t g0 = t * kMsTile;
    const int64_t g1 = min(total, g0 + kMsTile);
    const int64_t p0 = g0 + static_cast<int64_t>(threadIdx.x) * kMsItems;
    const int64_t tn = t + gridDim.x;
    int2 prn = pr;
    int64_t rbn = 0;
    if (tn < ntiles) {
      ms_load_tile<false>(col, nullptr, tn * kMsTile + static_cast<int64_t>(threadIdx.x) * kMsItems,
                          min(total, (tn + 1) * kMsTile), cn, unused);
      prn = part[tn];
      if (threadIdx.x <= min(gr, static_cast<int64_t>(prn.y - prn.x + 1))) rbn = rp[prn.x + threadIdx.x];
    }
    for (int64_t w0 = pr.x; w0 <= pr.y; w0 += gr) {  // windows of at most gr rows
      const int nr = static_cast<int>(min(gr, static_cast<int64_t>(pr.y) - w0 + 1));
      if (w0 == pr.x && nr < static_cast<int>(blockDim.x)) {
        if (threadIdx.x <= nr) rstart[threadIdx.x] = rb;
      } else {
        for (int i = threadIdx.x; i <= nr; i += blockDim.x) rstart[i] = rp[w0 + i];
      }
      for (int64_t i = threadIdx.x; i < nr * v; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      int bin[kMsItems];
      ms_bins(rstart, nr, p0, g1, c, shift, v, bin, err);
#pragma unroll
      for (int j = 0; j < kMsItems; ++j) ms_count<MATCH>(hist, bin[j]);
      __syncthreads();
      for (int64_t b = threadIdx.x; b < nr * v; b += blockDim.x) {
        const unsigned h = hist[b];
        if (h) atomicAdd(&counts[(w0 + b / v) * v + (b % v)], static_cast<unsigned long long>(h));
      }
      __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < kMsItems; ++j) c[j] = cn[j];
    pr = prn;
    rb = rbn;
  }
}

void launch_histogram(const int64_t* row_ptr, const int2* part, int64_t total, const int32_t* col, int shift,
                      int64_t nchunks, int64_t group_rows, unsigned long long* counts, bool match, int sms,
                      uint32_t* err, cudaStream_t s) {
  if (total == 0) return;
  const size_t smem = (group_rows + 1) * 8 + group_rows * nchunks * 4;
  const int64_t ntiles = ceil_div(total, kMsTile);
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(ntiles, static_cast<int64_t>(sms) * 4));
  if (match) {
    cudaFuncSetAttribute(k_histogram<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    note_launch();
    k_histogram<true><<<grid, kMsThreads, smem, s>>>(row_ptr, part, total, ntiles, col, shift, nchunks, group_rows,
                                                     counts, err);
  } else {
    cudaFuncSetAttribute(k_histogram<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    note_launch();
    k_histogram<false><<<grid, kMsThreads, smem, s>>>(row_ptr, part, total, ntiles, col, shift, nchunks, group_rows,
                                                      counts, err);
  }
}

// Small blocks (128 threads, eight per SM) keep the phases of many tiles in flight at once:
// the tile load, the counting, the reservations and the scatter of different blocks overlap.
// Measured on R-MAT scale 18 with 512 / 256 / 128 / 64 / 32 threads per block: 14.4 / 13.3 /
// 12.6 / 12.4 / 19.5 ms (the smallest tiles drown in global reservations).
template <bool VALS, bool MATCH>
__global__ void __launch_bounds__(kMsThreads, 8) k_multisplit(
    const int64_t* __restrict__ rp, const int2* __restrict__ part, int64_t total, int64_t ntiles,
    const int32_t* __restrict__ in_col, const double* __restrict__ in_val, int shift, int64_t v, int64_t gr,
    const int32_t* __restrict__ xmap, unsigned long long* __restrict__ cursor, int32_t* __restrict__ out_col,
    double* __restrict__ out_val, uint32_t* err) {
  extern __shared__ __align__(16) char smem_raw[];
  unsigned long long* goff = reinterpret_cast<unsigned long long*>(smem_raw);  // gr*v: global run starts
  int64_t* rstart = reinterpret_cast<int64_t*>(goff + gr * v);                 // gr + 1
  unsigned* hist = reinterpret_cast<unsigned*>(rstart + gr + 1);               // gr*v
  const int64_t wmask = (int64_t(1) << shift) - 1;
  int64_t t = blockIdx.x;
  if (t >= ntiles) return;
  int32_t c[kMsItems];
  double vv[kMsItems];
  ms_load_tile<VALS>(in_col, in_val, t * kMsTile + static_cast<int64_t>(threadIdx.x) * kMsItems,
                     min(total, (t + 1) * kMsTile), c, vv);
  int2 pr = part[t];
  for (; t < ntiles; t += gridDim.x) {
    const int64_t g0 = t * kMsTile;
    const int64_t g1 = min(total, g0 + kMsTile);
    const int64_t p0 = g0 + static_cast<int64_t>(threadIdx.x) * kMsItems;
    const int64_t tn = t + gridDim.x;
    for (int64_t w0 = pr.x; w0 <= pr.y; w0 += gr) {
      const int nr = static_cast<int>(min(gr, static_cast<int64_t>(pr.y) - w0 + 1));
      const int nbins = static_cast<int>(nr * v);
      for (int i = threadIdx.x; i <= nr; i += blockDim.x) rstart[i] = rp[w0 + i];
      for (int i = threadIdx.x; i < nbins; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      int bin[kMsItems];
      unsigned rank[kMsItems];
      ms_bins(rstart, nr, p0, g1, c, shift, v, bin, err);
#pragma unroll
      for (int j = 0; j < kMsItems; ++j) rank[j] = ms_rank<MATCH>(hist, bin[j]);
      __syncthreads();
      // one global reservation per bin: its run of the bin's chunk in C^_reord
      {
        const int per = (nbins + kMsThreads - 1) / kMsThreads;
        const int b0 = threadIdx.x * per;
        for (int b = b0; b < min(nbins, b0 + per); ++b) {
          const unsigned h = hist[b];
          if (h) {
            const int64_t gchunk = (w0 + b / v) * v + (b % v);
            const int64_t q = xmap ? xmap[gchunk] : gchunk;
            goff[b] = atomicAdd(&cursor[q], static_cast<unsigned long long>(h));
          }
        }
      }
      __syncthreads();
      // scatter: every element goes straight to its bin's reserved run (run start + rank).  A
      // bin's run is written by this block alone within this tile, so the partial sectors of
      // neighbouring lanes merge in L2 and DRAM sees whole lines (no permute in shared memory)
#pragma unroll
      for (int j = 0; j < kMsItems; ++j) {
        const int b = bin[j];
        if (b >= 0) {
          const int64_t dst = static_cast<int64_t>(goff[b]) + rank[j];
          __stcs(&out_col[dst], static_cast<int32_t>(c[j] & wmask));
          if (VALS) __stcs(&out_val[dst], vv[j]);
        }
      }
      // no barrier here: the next window's first barrier orders the reuse of hist and goff
      if (w0 + gr > pr.y && tn < ntiles)
        ms_load_tile<VALS>(in_col, in_val, tn * kMsTile + static_cast<int64_t>(threadIdx.x) * kMsItems,
                           min(total, (tn + 1) * kMsTile), c, vv);
    }
    if (tn < ntiles) pr = part[tn];
  }
}

template <bool VALS, bool MATCH>
static void ms_launch(const int64_t* row_ptr, const int2* part, int64_t total, const int32_t* in_col,
                      const double* in_val, int shift, int64_t nchunks, int64_t group_rows, const int32_t* xmap,
                      unsigned long long* cursor, int32_t* out_col, double* out_val, int sms, uint32_t* err,
                      cudaStream_t s) {
  const int64_t bins = group_rows * nchunks;
  const size_t smem = bins * 8 + (group_rows + 1) * 8 + bins * 4;
  const int64_t ntiles = ceil_div(total, kMsTile);
  auto kern = k_multisplit<VALS, MATCH>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kMsThreads, smem);
  if (per_sm < 1) per_sm = 1;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(ntiles, static_cast<int64_t>(sms) * per_sm));
  note_launch();
  kern<<<grid, kMsThreads, smem, s>>>(row_ptr, part, total, ntiles, in_col, in_val, shift, nchunks, group_rows, xmap,
                                      cursor, out_col, out_val, err);
}

void launch_multisplit(const int64_t* row_ptr, const int2* part, int64_t total, const int32_t* in_col,
                       const double* in_val, int shift, int64_t nchunks, int64_t group_rows, const int32_t* xmap,
                       unsigned long long* reord_cursor, int32_t* out_col, double* out_val, bool with_vals, bool match,
                       int sms, uint32_t* err, cudaStream_t s) {
  if (total == 0) return;
  if (with_vals) {
    if (match) ms_launch<true, true>(row_ptr, part, total, in_col, in_val, shift, nchunks, group_rows, xmap,
                                     reord_cursor, out_col, out_val, sms, err, s);
    else ms_launch<true, false>(row_ptr, part, total, in_col, in_val, shift, nchunks, group_rows, xmap,
                                reord_cursor, out_col, out_val, sms, err, s);
  } else {
    if (match) ms_launch<false, true>(row_ptr, part, total, in_col, nullptr, shift, nchunks, group_rows, xmap,
                                      reord_cursor, out_col, nullptr, sms, err, s);
    else ms_launch<false, false>(row_ptr, part, total, in_col, nullptr, shift, nchunks, group_rows, xmap,
                                 reord_cursor, out_col, nullptr, sms, err, s);
  }
}

// ---- chunk partition, metadata and final chunk descriptors ---------------------------------------
__global__ void k_chunk_partition(const unsigned long long* __restrict__ counts, int64_t n, int64_t tau,
                                  uint8_t* __restrict__ bin) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) bin[i] = counts[i] > static_cast<unsigned long long>(tau) ? 0 : 1;
}
void launch_chunk_partition(const unsigned long long* counts, int64_t n, int64_t tau, uint8_t* bin,
                            cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_chunk_partition<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0, s>>>(counts, n, tau, bin);
}

__global__ void k_invert(const int32_t* __restrict__ list, int64_t n, int32_t* __restrict__ xmap) {
  const int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (q < n) xmap[list[q]] = static_cast<int32_t>(q);
}
void launch_invert(const int32_t* list, int64_t n, int32_t* xmap, cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_invert<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0, s>>>(list, n, xmap);
}

__global__ void k_reord_meta(const unsigned long long* __restrict__ counts, int64_t nin, int64_t v,
                             const int32_t* __restrict__ xmap, const int32_t* __restrict__ in_row,
                             const int32_t* __restrict__ in_base, int64_t width, int64_t* __restrict__ rcnt,
                             int32_t* __restrict__ out_row, int32_t* __restrict__ out_base) {
  const int64_t id = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (id >= nin * v) return;
  const int64_t p = id / v, c = id % v;
  const int64_t q = xmap ? xmap[id] : id;
  rcnt[q] = static_cast<int64_t>(counts[id]);
  out_row[q] = in_row ? in_row[p] : static_cast<int32_t>(p);
  out_base[q] = (in_base ? in_base[p] : 0) + static_cast<int32_t>(c * width);
}
void launch_reord_meta(const unsigned long long* counts, int64_t nrows_in, int64_t nchunks, const int32_t* xmap,
                       const int32_t* in_row, const int32_t* in_base, int64_t width, int64_t* reord_cnt,
                       int32_t* out_row, int32_t* out_base, cudaStream_t s) {
  const int64_t n = nrows_in * nchunks;
  if (n == 0) return;
  note_launch();
  k_reord_meta<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0, s>>>(counts, nrows_in, nchunks, xmap, in_row,
                                                                       in_base, width, reord_cnt, out_row, out_base);
}

__global__ void k_final_desc(const int64_t* __restrict__ rptr, int64_t q0, int64_t q1, int64_t elem_base,
                             const int32_t* __restrict__ row, const int32_t* __restrict__ base,
                             int64_t* __restrict__ fs, int64_t* __restrict__ fc, int32_t* __restrict__ fr,
                             int32_t* __restrict__ fb) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t q = q0 + i;
  if (q >= q1) return;
  fs[i] = elem_base + rptr[q];
  fc[i] = rptr[q + 1] - rptr[q];
  fr[i] = row ? row[q] : static_cast<int32_t>(q);
  fb[i] = base ? base[q] : 0;
}
void launch_final_desc(const int64_t* reord_ptr, int64_t q0, int64_t q1, int64_t elem_base, const int32_t* row,
                       const int32_t* base, int64_t* f_start, int64_t* f_cnt, int32_t* f_row, int32_t* f_base,
                       cudaStream_t s) {
  if (q1 <= q0) return;
  note_launch();
  k_final_desc<<<static_cast<unsigned>(ceil_div(q1 - q0, 256)), 256, 0, s>>>(reord_ptr, q0, q1, elem_base, row,
                                                                             base, f_start, f_cnt, f_row, f_base);
}

// Accumulator bin of a final chunk.  Chunks of the last level (width W, bitmap kernels):
// bins nlad + 0..3 = hash for <= 256 elements (warp), <= 1024, <= kChunkDenseMin, and the
// dense accumulator above.  Light chunks of earlier levels (wider, at most tau elements): the
// hash ladder levels 0..nlad-1 of the row accumulators.
__global__ void k_chunk_classify(const int64_t* __restrict__ fc, int64_t n, int64_t bitmap_from, BinRule r,
                                 uint8_t* __restrict__ bin) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t c = fc[i];
  uint8_t b;
  if (c == 0) {
    b = kBinEmpty;
  } else if (i >= bitmap_from) {
    b = static_cast<uint8_t>(r.n + (c <= kWarpChunkMax ? 0 : (c <= kBlockChunkMax ? 1 : (c <= kChunkDenseMin ? 2 : 3))));
  } else {
    int L = 0;
    while (L < r.n - 1 && c > r.upper[L]) ++L;
    b = static_cast<uint8_t>(L);
  }
  bin[i] = b;
}
void launch_chunk_classify(const int64_t* f_cnt, int64_t n, int64_t bitmap_from, const BinRule& rule,
                           uint8_t* bin, cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_chunk_classify<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0, s>>>(f_cnt, n, bitmap_from, rule, bin);
}

// Offsets of the final chunks inside their C rows: a dense grid (row, finest chunk) of
// chunk sizes, scanned; chunk offset = grid prefix at the chunk - grid prefix at the row start.
__global__ void k_grid_fill(const int32_t* __restrict__ fr, const int32_t* __restrict__ fb,
                            const int64_t* __restrict__ fnnz, int64_t n, int shift, int64_t nfin,
                            int64_t* __restrict__ grid) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) grid[static_cast<int64_t>(fr[i]) * nfin + (fb[i] >> shift)] = fnnz[i];
}
void launch_grid_fill(const int32_t* f_row, const int32_t* f_base, const int64_t* f_nnz, int64_t n, int shift_fin,
                      int64_t nfin, int64_t* grid, cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_grid_fill<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0, s>>>(f_row, f_base, f_nnz, n, shift_fin, nfin,
                                                                      grid);
}
__global__ void k_grid_finish(const int64_t* __restrict__ S, const int32_t* __restrict__ fr,
                              const int32_t* __restrict__ fb, int64_t n, int shift, int64_t nfin,
                              int64_t* __restrict__ fout) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) {
    const int64_t r0 = static_cast<int64_t>(fr[i]) * nfin;
    fout[i] = S[r0 + (fb[i] >> shift)] - S[r0];
  }
}
void launch_grid_finish(const int64_t* grid_scanned, const int32_t* f_row, const int32_t* f_base, int64_t n,
                        int shift_fin, int64_t nfin, int64_t* f_out, cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_grid_finish<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0, s>>>(grid_scanned, f_row, f_base, n,
                                                                        shift_fin, nfin, f_out);
}
__global__ void k_row_totals(const int64_t* __restrict__ S, int64_t nrows, int64_t nfin,
                             const int32_t* __restrict__ rows, int64_t* __restrict__ row_nnz) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r < nrows) row_nnz[rows[r]] = S[(r + 1) * nfin] - S[r * nfin];
}
void launch_row_totals(const int64_t* grid_scanned, int64_t nrows, int64_t nfin, const int32_t* heavy_rows,
                       int64_t* row_nnz, cudaStream_t s) {
  if (nrows == 0) return;
  note_launch();
  k_row_totals<<<static_cast<unsigned>(ceil_div(nrows, 256)), 256, 0, s>>>(grid_scanned, nrows, nfin, heavy_rows,
                                                                           row_nnz);
}

}  // namespace sg
