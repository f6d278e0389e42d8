// Long rows by a hash accumulator in shared and global memory (SPGEMM_FLAG_LONG_ROWS), after the
// Ocean page's hybrid accumulator: rows too long for one SM's hash table are accumulated by one
// block each in a shared-memory table that spills into a global-memory table of the row.  It
// replaces, for the heavy rows, the outer product + multisplit + chunk accumulators of the
// gMAGNUS pipeline, so the two routes for rows that overflow on-chip accumulators can be compared
// on the same inputs.
//
//   * A block takes a heavy row (persistent blocks, rows in turn); its warps take the row's
//     entries A[r,k] in turn and sweep row k of B with their lanes (Gustavson's order).
//   * A product's column probes kLongProbe slots of the block's shared table (linear probing,
//     keys claimed by CAS, values summed by shared atomics); when all of them hold other columns
//     it moves to the row's global table (probing to the end; global atomics).  Slots are never
//     freed, so every column lives in exactly one of the two tables.
//   * Symbolic: the count of columns claimed, the row's nnz.
//   * Numeric: every occupied slot sets its column's bit in a bitmap of the row's columns
//     (global, one per block); a block scan of the words' popcounts ranks every column (set
//     bits below it), and each entry is written at its final position: the row comes out sorted
//     without sorting.  The page's own kernel sorts the hash entries instead (indirect key/ptr
//     radix sort); ranking through the bitmap does the same in one pass.
#include <algorithm>

#include "internal.h"

namespace sg {

namespace {

constexpr int kLongThreads = 1024;
constexpr int kLongSlots = 8192;   // shared slots per block: keys 32 KB (+ values 64 KB in numeric)
constexpr int kLongProbe = 16;     // shared probes before a column moves to the row's global table

struct LongParams {
  const int64_t* arp;
  const int32_t* acol;
  const double* aval;
  const int64_t* brp;
  const int32_t* bcol;
  const double* bval;
  const int32_t* rows;   // the group's heavy rows (global row ids)
  int64_t nrows;
  const int64_t* goff;   // nrows + 1: global table of row j = slots [goff[j], goff[j+1]) - gbase (power of two)
  int64_t gbase;
  int32_t* gkeys;
  double* gvals;         // numeric
  uint32_t* gbits;       // numeric: per block, nwords bitmap words then nwords prefix words
  int64_t nwords;
  Sink sink;
  uint32_t* err;
};

template <bool NUM>
__device__ __forceinline__ bool long_insert(int32_t* skeys, double* svals, int32_t* gk, double* gv, uint32_t gcap,
                                            int32_t col, double v, uint32_t* err) {
  uint32_t slot = hash_slot(col, kLongSlots);
#pragma unroll 1
  for (int probe = 0; probe < kLongProbe; ++probe) {
    const int32_t k = *reinterpret_cast<volatile int32_t*>(&skeys[slot]);
    if (k == col) {
      if (NUM) atomicAdd(&svals[slot], v);
      return false;
    }
    if (k == kEmptyKey) {
      const int32_t old = atomicCAS(&skeys[slot], kEmptyKey, col);
      if (old == kEmptyKey || old == col) {
        if (NUM) atomicAdd(&svals[slot], v);
        return old == kEmptyKey;
      }
    }
    slot = (slot + 1) & (kLongSlots - 1);
  }
  uint32_t gs = hash_slot(col, gcap);
  for (uint32_t probe = 0; probe < gcap; ++probe) {
    const int32_t k = *reinterpret_cast<volatile int32_t*>(&gk[gs]);
    if (k == col) {
      if (NUM) atomicAdd(&gv[gs], v);
      return false;
    }
    if (k == kEmptyKey) {
      const int32_t old = atomicCAS(&gk[gs], kEmptyKey, col);
      if (old == kEmptyKey || old == col) {
        if (NUM) atomicAdd(&gv[gs], v);
        return old == kEmptyKey;
      }
    }
    gs = (gs + 1 == gcap) ? 0 : gs + 1;
  }
  set_error(err, kErrHashFull);
  return false;
}

// Rank of column c through the bitmap and its word prefix.
__device__ __forceinline__ int64_t long_rank(const uint32_t* bits, const uint32_t* pre, int32_t c) {
  return static_cast<int64_t>(pre[c >> 5]) + __popc(bits[c >> 5] & ((1u << (c & 31)) - 1u));
}

template <bool NUM>
__global__ void __launch_bounds__(kLongThreads, 1) k_long(LongParams p) {
  extern __shared__ __align__(16) char smem_raw[];
  __shared__ int64_t red[33];
  __shared__ unsigned long long s_count;
  int32_t* skeys = reinterpret_cast<int32_t*>(smem_raw);
  double* svals = reinterpret_cast<double*>(smem_raw + sizeof(int32_t) * kLongSlots);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  uint32_t* bits = NUM ? p.gbits + static_cast<int64_t>(blockIdx.x) * 2 * p.nwords : nullptr;
  uint32_t* pre = NUM ? bits + p.nwords : nullptr;
  for (int64_t j = blockIdx.x; j < p.nrows; j += gridDim.x) {
    const int64_t row = p.rows[j];
    const bool in_window = !NUM || (row >= p.sink.row_begin && row < p.sink.row_end);
    if (!in_window) continue;  // uniform over the block
    const int64_t g0 = p.goff[j] - p.gbase;
    const uint32_t gcap = static_cast<uint32_t>(p.goff[j + 1] - p.goff[j]);
    int32_t* gk = p.gkeys + g0;
    double* gv = NUM ? p.gvals + g0 : nullptr;
    for (int i = threadIdx.x; i < kLongSlots; i += blockDim.x) {
      skeys[i] = kEmptyKey;
      if (NUM) svals[i] = 0.0;
    }
    for (uint32_t i = threadIdx.x; i < gcap; i += blockDim.x) {
      gk[i] = kEmptyKey;
      if (NUM) gv[i] = 0.0;
    }
    if (NUM)
      for (int64_t w = threadIdx.x; w < p.nwords; w += blockDim.x) bits[w] = 0u;
    if (threadIdx.x == 0) s_count = 0;
    __syncthreads();
    // expansion: warps take the row's entries in turn, lanes sweep the B row
    unsigned long long fresh = 0;
    const int64_t a0 = p.arp[row], a1 = p.arp[row + 1];
    for (int64_t e = a0 + warp; e < a1; e += nwarps) {
      const int32_t k = p.acol[e];
      const double a = NUM ? p.aval[e] : 0.0;
      const int64_t b1 = p.brp[k + 1];
      for (int64_t q = p.brp[k] + lane; q < b1; q += 32) {
        const int32_t c = p.bcol[q];
        if (c < 0 || (static_cast<int64_t>(c) >> 5) >= p.nwords) {
          set_error(p.err, kErrBounds);
          continue;
        }
        fresh += long_insert<NUM>(skeys, svals, gk, gv, gcap, c, NUM ? a * p.bval[q] : 0.0, p.err);
      }
    }
    fresh = warp_sum(fresh);
    if (lane == 0) atomicAdd(&s_count, fresh);
    __syncthreads();
    const int64_t nnz = static_cast<int64_t>(s_count);
    if (!NUM) {
      if (threadIdx.x == 0) p.sink.row_nnz[row] = nnz;
      __syncthreads();
      continue;
    }
    // numeric: bitmap of the row's columns, word prefix, ranked write
    for (int i = threadIdx.x; i < kLongSlots; i += blockDim.x) {
      const int32_t c = skeys[i];
      if (c != kEmptyKey) atomicOr(&bits[c >> 5], 1u << (c & 31));
    }
    for (uint32_t i = threadIdx.x; i < gcap; i += blockDim.x) {
      const int32_t c = gk[i];
      if (c != kEmptyKey) atomicOr(&bits[c >> 5], 1u << (c & 31));
    }
    __syncthreads();
    {
      const int64_t per = ceil_div(p.nwords, static_cast<int64_t>(blockDim.x));
      const int64_t w0 = threadIdx.x * per, w1 = min(p.nwords, w0 + per);
      int64_t local = 0;
      for (int64_t w = w0; w < w1; ++w) local += __popc(bits[w]);
      int64_t total;
      const int64_t incl = block_incl_scan(local, red, &total);
      int64_t run = incl - local;
      for (int64_t w = w0; w < w1; ++w) {
        pre[w] = static_cast<uint32_t>(run);
        run += __popc(bits[w]);
      }
      if (total != nnz || total != p.sink.row_ptr[row + 1] - p.sink.row_ptr[row]) {
        if (threadIdx.x == 0) set_error(p.err, kErrRowOverflow);
      }
    }
    __syncthreads();
    const int64_t expected = p.sink.row_ptr[row + 1] - p.sink.row_ptr[row];
    const int64_t out = p.sink.row_ptr[row] - p.sink.row_ptr[p.sink.row_begin];
    int32_t* c_col = p.sink.c_col + out;
    double* c_val = p.sink.c_val + out;
    for (int i = threadIdx.x; i < kLongSlots; i += blockDim.x) {
      const int32_t c = skeys[i];
      if (c != kEmptyKey) {
        const int64_t r = long_rank(bits, pre, c);
        if (r < expected) {
          c_col[r] = c;
          c_val[r] = svals[i];
        }
      }
    }
    for (uint32_t i = threadIdx.x; i < gcap; i += blockDim.x) {
      const int32_t c = gk[i];
      if (c != kEmptyKey) {
        const int64_t r = long_rank(bits, pre, c);
        if (r < expected) {
          c_col[r] = c;
          c_val[r] = gv[i];
        }
      }
    }
    __syncthreads();
  }
}

}  // namespace

size_t long_smem_bytes(bool numeric) {
  return static_cast<size_t>(kLongSlots) * (sizeof(int32_t) + (numeric ? sizeof(double) : 0));
}

int long_blocks(int sms) { return 2 * sms; }

void launch_long(const spgemm_csr& A, const spgemm_csr& B, const int32_t* rows, int64_t nrows, const int64_t* goff,
                 int64_t gbase, int32_t* gkeys, double* gvals, uint32_t* gbits, int64_t nwords, bool numeric,
                 const Sink& sink, int blocks, uint32_t* err, cudaStream_t s) {
  if (nrows == 0) return;
  LongParams p{};
  p.arp = A.row_ptr;
  p.acol = A.col_idx;
  p.aval = A.vals;
  p.brp = B.row_ptr;
  p.bcol = B.col_idx;
  p.bval = B.vals;
  p.rows = rows;
  p.nrows = nrows;
  p.goff = goff;
  p.gbase = gbase;
  p.gkeys = gkeys;
  p.gvals = gvals;
  p.gbits = gbits;
  p.nwords = nwords;
  p.sink = sink;
  p.err = err;
  const size_t smem = long_smem_bytes(numeric);
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(nrows, blocks));
  note_launch();
  if (numeric) {
    cudaFuncSetAttribute(k_long<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    k_long<true><<<grid, kLongThreads, smem, s>>>(p);
  } else {
    cudaFuncSetAttribute(k_long<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    k_long<false><<<grid, kLongThreads, smem, s>>>(p);
  }
}

// Global table slots of every listed row: the power of two at least twice its bound (IP in the
// symbolic phase, nnz in the numeric one), at least 64.
__global__ void k_long_caps(const int32_t* __restrict__ rows, int64_t n, const int64_t* __restrict__ bound,
                            const int64_t* __restrict__ row_ptr, int64_t* __restrict__ cap) {
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j >= n) return;
  const int64_t r = rows[j];
  const int64_t b = row_ptr ? row_ptr[r + 1] - row_ptr[r] : bound[r];
  int64_t c = 64;
  while (c < 2 * b) c <<= 1;
  cap[j] = c;
}
void launch_long_caps(const int32_t* rows, int64_t n, const int64_t* ip, const int64_t* row_ptr, int64_t* cap,
                      cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_long_caps<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0, s>>>(rows, n, ip, row_ptr, cap);
}

}  // namespace sg
