// Shared-memory accumulators (gMAGNUS page, sections II-B and III-E):
//   * light rows of C: Gustavson expansion of row i (every A[i,k] scales row k of B), summed
//     in a hash map (modulo hashing, linear probing, load factor 1/2) or, when the row's
//     column span is narrow, in a shortened dense array over that span;
//   * final chunks of C^_reord: a flat list of (local column, value) pairs, summed in a hash
//     map (light chunks) or in a dense array of the chunk width plus a bitmap (heavy chunks).
// Symbolic phase: count the distinct columns.  Numeric phase: accumulate, then produce the
// row (or chunk) sorted by column -- a bitonic sort of the compacted hash entries, or a scan
// over the dense bitmap -- and write it at its final CSR position.
//
// One group of threads owns one row or chunk: a warp (several per block) for small bins, a
// whole block for large ones (bin ladder after the Ocean page, section 4: each larger kernel
// doubles the threads and the accumulator).
#include "internal.h"

namespace sg {

constexpr int kWarpGroupsPerBlock = 8;
constexpr int kMaxBatch = 256;  // A entries staged per expansion step
constexpr int kExpandUnroll = 4;  // products per thread whose loads are issued together

struct AccParams {
  // row source
  const int64_t* arp;
  const int32_t* acol;
  const double* aval;
  const int64_t* brp;
  const int32_t* bcol;
  const double* bval;
  const int32_t* span_lo;
  // chunk source
  ChunkSet cs;
  // common
  const int32_t* list;
  int64_t count;
  int64_t slots;       // hash slots, or dense width
  Sink sink;
  uint32_t* err;
  int has_vals;        // chunk source carries values
  EstSink est;         // estimated workflows: capacities and the temporary output (numeric rows)
  int est_on;
};

template <bool WARP>
struct Group {
  int lane, size;
  __device__ __forceinline__ void sync() const {
    if (WARP) __syncwarp(); else __syncthreads();
  }
};

// Inclusive scan over the group; `tmp` is 33 int64 of shared memory (block groups only).
template <bool WARP>
__device__ __forceinline__ int64_t group_scan(const Group<WARP>& g, int64_t v, int64_t* tmp,
                                              int64_t* total) {
  if (WARP) {
    int64_t x = warp_incl_scan(v);
    *total = __shfl_sync(0xffffffffu, x, 31);
    return x;
  } else {
    return block_incl_scan(v, tmp, total);
  }
}

// 32-bit variant (tmp reinterpreted as 33 int32).
template <bool WARP>
__device__ __forceinline__ int group_scan_i32(const Group<WARP>& g, int v, int64_t* tmp, int* total) {
  if (WARP) {
    const int x = warp_incl_scan(v);
    *total = __shfl_sync(0xffffffffu, x, 31);
    return x;
  } else {
    return block_incl_scan(v, reinterpret_cast<int*>(tmp), total);
  }
}

// Shared-memory layout of one group.
struct Smem {
  double* av;        // [batch] A values of the staged entries
  int64_t* bstart;   // [batch] first B index of the staged entries
  int32_t* incl;     // [batch] inclusive prefix of their B row lengths (a light row has at most
                     //         tau products, far below 2^31)
  int64_t* tmp;      // [34] scan scratch; word 33: overflow flag of the estimated workflows
  double* vals;      // [slots] (numeric)
  int32_t* keys;     // [slots] hash keys, or dense bitmap words
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

__host__ __device__ inline int batch_of(int size) { return size < kMaxBatch ? size : kMaxBatch; }

__host__ __device__ inline size_t group_bytes(int64_t slots, int size, bool dense, bool numeric,
                                              bool rows) {
  size_t b = align16(34 * sizeof(int64_t));
  if (rows) b += align16(batch_of(size) * (sizeof(double) + sizeof(int64_t) + sizeof(int32_t)));
  if (numeric) b += align16(static_cast<size_t>(slots) * sizeof(double));
  b += dense ? align16(((slots + 31) / 32) * sizeof(int32_t))
             : align16(static_cast<size_t>(slots) * sizeof(int32_t));
  return b;
}

__device__ __forceinline__ Smem carve(char* p, int64_t slots, int size, bool dense, bool numeric,
                                      bool rows) {
  Smem s;
  s.tmp = reinterpret_cast<int64_t*>(p);
  p += align16(34 * sizeof(int64_t));
  if (rows) {
    const int nb = batch_of(size);
    s.av = reinterpret_cast<double*>(p);
    s.bstart = reinterpret_cast<int64_t*>(p + nb * sizeof(double));
    s.incl = reinterpret_cast<int32_t*>(p + nb * (sizeof(double) + sizeof(int64_t)));
    p += align16(nb * (sizeof(double) + sizeof(int64_t) + sizeof(int32_t)));
  } else {
    s.av = nullptr;
    s.bstart = nullptr;
    s.incl = nullptr;
  }
  if (numeric) {
    s.vals = reinterpret_cast<double*>(p);
    p += align16(static_cast<size_t>(slots) * sizeof(double));
  } else {
    s.vals = nullptr;
  }
  s.keys = reinterpret_cast<int32_t*>(p);
  return s;
}

// ---- accumulators ------------------------------------------------------------------------
template <bool NUMERIC>
__device__ __forceinline__ bool hash_insert(const Smem& s, uint32_t slots, int32_t col, double v,
                                            uint32_t* err) {
  uint32_t slot = hash_slot(col, slots);
  for (uint32_t probe = 0; probe < slots; ++probe) {
    int32_t k = *reinterpret_cast<volatile int32_t*>(&s.keys[slot]);
    if (k == col) {
      if (NUMERIC) atomicAdd(&s.vals[slot], v);
      return false;
    }
    if (k == kEmptyKey) {
      const int32_t old = atomicCAS(&s.keys[slot], kEmptyKey, col);
      if (old == kEmptyKey || old == col) {
        if (NUMERIC) atomicAdd(&s.vals[slot], v);
        return old == kEmptyKey;
      }
    }
    slot = (slot + 1 == slots) ? 0 : slot + 1;
  }
  set_error(err, kErrHashFull);
  return false;
}

template <bool NUMERIC>
__device__ __forceinline__ bool dense_insert(const Smem& s, uint32_t width, int32_t idx, double v,
                                             uint32_t* err) {
  if (static_cast<uint32_t>(idx) >= width) {
    set_error(err, kErrBounds);
    return false;
  }
  const uint32_t bit = 1u << (idx & 31);
  const uint32_t old = atomicOr(reinterpret_cast<uint32_t*>(&s.keys[idx >> 5]), bit);
  if (NUMERIC) atomicAdd(&s.vals[idx], v);
  return (old & bit) == 0;
}

template <bool WARP, bool NUMERIC, bool DENSE>
__device__ __forceinline__ void acc_clear(const Group<WARP>& g, const Smem& s, int64_t slots) {
  if (DENSE) {
    const int64_t words = (slots + 31) / 32;
    for (int64_t w = g.lane; w < words; w += g.size) s.keys[w] = 0;
    if (NUMERIC)
      for (int64_t j = g.lane; j < slots; j += g.size) s.vals[j] = 0.0;
  } else {
    for (int64_t j = g.lane; j < slots; j += g.size) s.keys[j] = kEmptyKey;
    if (NUMERIC)
      for (int64_t j = g.lane; j < slots; j += g.size) s.vals[j] = 0.0;
  }
}

// ---- sources -----------------------------------------------------------------------------
// Expand row `row` of A*B into the accumulator; returns this thread's count of new columns.
// `ierr` receives hash-table overflows: the global error word, or (estimated workflows) the
// row's own flag, which also ends the expansion early.
template <bool WARP, bool NUMERIC, bool DENSE>
__device__ __forceinline__ int64_t expand_row(const Group<WARP>& g, const Smem& s,
                                              const AccParams& p, int64_t row, int32_t base,
                                              uint32_t slots, uint32_t* ierr) {
  int64_t fresh = 0;
  const int64_t a0 = p.arp[row], a1 = p.arp[row + 1];
  const int nb = batch_of(g.size);
  for (int64_t eb = a0; eb < a1; eb += nb) {
    const int nent = static_cast<int>(min(static_cast<int64_t>(nb), a1 - eb));
    int len = 0;
    if (g.lane < nent) {
      const int64_t e = eb + g.lane;
      const int32_t k = p.acol[e];
      const int64_t b0 = p.brp[k];
      len = static_cast<int>(p.brp[k + 1] - b0);
      s.av[g.lane] = NUMERIC ? p.aval[e] : 0.0;
      s.bstart[g.lane] = b0;
    }
    int total;
    const int incl = group_scan_i32<WARP>(g, g.lane < nb ? len : 0, s.tmp, &total);
    if (g.lane < nent) s.incl[g.lane] = incl;
    g.sync();
    int j = 0;
    // kExpandUnroll products per thread per step: their B loads are all issued before the
    // first accumulator update, so each thread keeps several L2 requests in flight
    for (int f0 = g.lane; f0 < total; f0 += kExpandUnroll * g.size) {
      if (ierr != p.err && *reinterpret_cast<volatile uint32_t*>(ierr) != 0u) break;  // row overflowed
      int32_t col[kExpandUnroll];
      double bv[kExpandUnroll], av[kExpandUnroll];
#pragma unroll
      for (int u = 0; u < kExpandUnroll; ++u) {
        const int f = f0 + u * g.size;
        col[u] = kEmptyKey;
        if (f < total) {
          // staged entry j holds flattened positions [incl[j-1], incl[j])
          if (s.incl[j] <= f) {
            int lo = j, hi = nent - 1;
            while (lo < hi) {
              const int mid = (lo + hi) >> 1;
              if (s.incl[mid] <= f) lo = mid + 1; else hi = mid;
            }
            j = lo;
          }
          const int before = j > 0 ? s.incl[j - 1] : 0;
          const int64_t q = s.bstart[j] + (f - before);
          col[u] = p.bcol[q];
          if (NUMERIC) {
            bv[u] = p.bval[q];
            av[u] = s.av[j];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kExpandUnroll; ++u) {
        if (col[u] == kEmptyKey) continue;
        const double v = NUMERIC ? av[u] * bv[u] : 0.0;
        if (DENSE) fresh += dense_insert<NUMERIC>(s, slots, col[u] - base, v, p.err);
        else fresh += hash_insert<NUMERIC>(s, slots, col[u], v, ierr);
      }
    }
    g.sync();
  }
  return fresh;
}

template <bool WARP, bool NUMERIC, bool DENSE>
__device__ __forceinline__ int64_t expand_chunk(const Group<WARP>& g, const Smem& s,
                                                const AccParams& p, int64_t start, int64_t cnt,
                                                uint32_t slots) {
  int64_t fresh = 0;
  const int32_t* col = p.cs.col + start;
  const double* val = p.cs.val + start;
  for (int64_t f = g.lane; f < cnt; f += g.size) {
    const int32_t c = col[f];
    const double v = (NUMERIC && p.has_vals) ? val[f] : 0.0;
    if (DENSE) fresh += dense_insert<NUMERIC>(s, slots, c, v, p.err);
    else fresh += hash_insert<NUMERIC>(s, slots, c, v, p.err);
  }
  return fresh;
}

// ---- outputs -----------------------------------------------------------------------------
// Block-wide exclusive prefix of n unsigned counters, in place.  Each warp owns a contiguous run
// of counters (read lane-strided, without bank conflicts) and scans it with shuffles; one
// barrier exchanges the run totals.  `tmp` holds 32 unsigned.  Ends with a barrier.
__device__ void block_exclusive_scan_inplace(const Group<false>& g, unsigned* a, int64_t n, unsigned* tmp) {
  const int nwarps = g.size >> 5, warp = g.lane >> 5, l = g.lane & 31;
  const int64_t per = ceil_div(ceil_div(n, nwarps), 32) * 32;
  const int64_t wb = warp * per, we = min(n, wb + per);
  unsigned c = 0;
  for (int64_t i = wb + l; i < we; i += 32) c += a[i];
  c = warp_sum(c);
  if (l == 0) tmp[warp] = c;
  __syncthreads();
  unsigned run = warp_sum(l < warp ? tmp[l] : 0u);
  for (int64_t i0 = wb; i0 < we; i0 += 32) {
    const int64_t i = i0 + l;
    const unsigned x = i < we ? a[i] : 0u;
    const unsigned incl = warp_incl_scan(x);
    if (i < we) a[i] = run + incl - x;
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  __syncthreads();
}

// Compact the occupied slots of a block's hash table to [0, n) in place; returns n.  The order
// is free (the ranked write orders by column).  Slabs of four slots per thread: a warp reads its
// 128 slots as four lane-strided rows, so every read of a slab precedes the barrier that
// releases its writes, and writes never reach past the slab.  The warp totals alternate between
// two halves of `tmp` (64 unsigned), so a fast warp cannot overwrite totals still being read.
__device__ int64_t block_compact(const Group<false>& g, const Smem& s, int64_t slots) {
  const int nwarps = g.size >> 5, warp = g.lane >> 5, l = g.lane & 31;
  unsigned* tmp = reinterpret_cast<unsigned*>(s.tmp);
  const int64_t slab = 128 * static_cast<int64_t>(nwarps);
  int64_t written = 0;
  int parity = 0;
  for (int64_t s0 = 0; s0 < slots; s0 += slab, parity ^= 1) {
    const int64_t b = s0 + 128 * warp + l;
    int32_t k[4];
    double v[4];
    unsigned occ[4], c = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t i = b + 32 * j;
      k[j] = i < slots ? s.keys[i] : kEmptyKey;
      v[j] = i < slots ? s.vals[i] : 0.0;
      occ[j] = __ballot_sync(0xffffffffu, k[j] != kEmptyKey);
      c += __popc(occ[j]);
    }
    unsigned* t = tmp + 32 * parity;
    if (l == 0) t[warp] = c;
    __syncthreads();
    const unsigned mine = l < warp ? t[l] : 0u;
    const unsigned all = l < nwarps ? t[l] : 0u;
    int64_t pos = written + warp_sum(mine);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (k[j] != kEmptyKey) {
        const int64_t d = pos + __popc(occ[j] & lanemask_lt());
        s.keys[d] = k[j];
        s.vals[d] = v[j];
      }
      pos += __popc(occ[j]);
    }
    written += warp_sum(all);
  }
  __syncthreads();
  return written;
}

// Ordered write of the `n` compacted entries [0, n) of a block's hash table without sorting, in
// a number of barriers independent of the row's column span.  When the span [lo, hi] fits one
// bitmap in the free part of the keys region, an entry's rank is the number of set bits below
// its column.  Otherwise: a counting sort of the entries into B >= n buckets of equal column
// width (B = the largest power of two not above the free slots, counters in the free keys
// region) and a rank inside the bucket by comparison with its few members.  Either way the
// entry index is scattered to its rank (index arrays in the free part of the values region:
// slots >= 2n leaves 2n free words there) and the write of C is coalesced.
__device__ void block_bucket_emit(const Group<false>& g, const Smem& s, int64_t slots, int64_t n, int64_t expected,
                                  int32_t col_base, int32_t* c_col, double* c_val, uint32_t* err) {
  if (n != expected) {
    if (g.lane == 0) set_error(err, kErrRowOverflow);
    return;
  }
  if (n == 0) return;
  int32_t lo = 0x7fffffff, hi = -1;
  for (int64_t i = g.lane; i < n; i += g.size) {
    lo = min(lo, s.keys[i]);
    hi = max(hi, s.keys[i]);
  }
  // block min / max through the scan scratch
  for (int d = 16; d > 0; d >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, d));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, d));
  }
  int32_t* red = reinterpret_cast<int32_t*>(s.tmp);
  if (lane_id() == 0) {
    red[2 * (threadIdx.x >> 5)] = lo;
    red[2 * (threadIdx.x >> 5) + 1] = hi;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int nw = (blockDim.x + 31) >> 5;
    int32_t a = threadIdx.x < nw ? red[2 * threadIdx.x] : 0x7fffffff;
    int32_t b = threadIdx.x < nw ? red[2 * threadIdx.x + 1] : -1;
    for (int d = 16; d > 0; d >>= 1) {
      a = min(a, __shfl_xor_sync(0xffffffffu, a, d));
      b = max(b, __shfl_xor_sync(0xffffffffu, b, d));
    }
    if (threadIdx.x == 0) {
      red[64] = a;
      red[65] = b;
    }
  }
  __syncthreads();
  lo = red[64];
  hi = red[65];
  __syncthreads();
  const int64_t span_words = (static_cast<int64_t>(hi) - lo) / 32 + 1;
  if (span_words <= slots - n) {
    // the row's column span fits one bitmap in the free keys region: rank = set bits below the
    // column (prefix of the word popcounts in the free values region)
    uint32_t* bits = reinterpret_cast<uint32_t*>(s.keys + n);        // span_words
    unsigned* pre = reinterpret_cast<unsigned*>(s.vals) + 2 * n;     // span_words
    int32_t* inv = reinterpret_cast<int32_t*>(pre + span_words);     // n (2n + span_words + n <= 2 slots)
    for (int64_t w = g.lane; w < span_words; w += g.size) bits[w] = 0u;
    __syncthreads();
    for (int64_t i = g.lane; i < n; i += g.size) {
      const int32_t c = s.keys[i] - lo;
      atomicOr(&bits[c >> 5], 1u << (c & 31));
    }
    __syncthreads();
    for (int64_t w = g.lane; w < span_words; w += g.size) pre[w] = __popc(bits[w]);
    __syncthreads();
    block_exclusive_scan_inplace(g, pre, span_words, reinterpret_cast<unsigned*>(s.tmp));
    for (int64_t i = g.lane; i < n; i += g.size) {
      const int32_t c = s.keys[i] - lo;
      inv[pre[c >> 5] + __popc(bits[c >> 5] & ((1u << (c & 31)) - 1u))] = static_cast<int32_t>(i);
    }
    __syncthreads();
    for (int64_t r = g.lane; r < n; r += g.size) {
      const int32_t i = inv[r];
      c_col[r] = s.keys[i] + col_base;
      c_val[r] = s.vals[i];
    }
    return;
  }
  int64_t nb = 1;  // buckets
  while (nb * 2 <= slots - n) nb *= 2;
  int shift = 0;    // bucket of a key: (key - lo) >> shift < nb
  while (((static_cast<int64_t>(hi) - lo) >> shift) >= nb) ++shift;
  unsigned* cnt = reinterpret_cast<unsigned*>(s.keys + n);      // nb counters
  int32_t* order = reinterpret_cast<int32_t*>(s.vals) + 2 * n;  // n entry indices, bucket by bucket
  int32_t* inv = order + n;                                     // n: entry index of each output position
  for (int64_t b = g.lane; b < nb; b += g.size) cnt[b] = 0u;
  __syncthreads();
  for (int64_t i = g.lane; i < n; i += g.size) atomicAdd(&cnt[(s.keys[i] - lo) >> shift], 1u);
  __syncthreads();
  block_exclusive_scan_inplace(g, cnt, nb, reinterpret_cast<unsigned*>(s.tmp));  // cnt[b]: start of bucket b
  for (int64_t i = g.lane; i < n; i += g.size)
    order[atomicAdd(&cnt[(s.keys[i] - lo) >> shift], 1u)] = static_cast<int32_t>(i);  // cnt[b]: end of bucket b
  __syncthreads();
  // rank inside the bucket, taken in bucket order: the lanes of a warp mostly share one bucket,
  // so they run the same number of comparisons and read the same members (broadcast loads); in
  // entry order one dense bucket would hold back every warp that has one of its members
  for (int64_t p = g.lane; p < n; p += g.size) {
    const int32_t i = order[p];
    const int32_t k = s.keys[i];
    const int64_t bk = (k - lo) >> shift;
    const unsigned b0 = bk > 0 ? cnt[bk - 1] : 0u, b1 = cnt[bk];
    unsigned r = b0;
    for (unsigned j = b0; j < b1; ++j) r += s.keys[order[j]] < k ? 1u : 0u;  // columns are distinct
    inv[r] = i;
  }
  __syncthreads();
  for (int64_t r = g.lane; r < n; r += g.size) {
    const int32_t i = inv[r];
    c_col[r] = s.keys[i] + col_base;
    c_val[r] = s.vals[i];
  }
}

// Sorted write of a hash table holding `n` entries: compact in place (rounds over the
// slots; every entry moves to a lower or equal slot), bitonic sort of the first 2^ceil(log2 n)
// slots, then a coalesced write.
template <bool WARP>
__device__ void hash_emit(const Group<WARP>& g, const Smem& s, int64_t slots, int64_t n,
                          int64_t expected, int32_t col_base, int32_t* c_col, double* c_val,
                          uint32_t* err) {
  if constexpr (!WARP) {
    const int64_t m = block_compact(g, s, slots);
    block_bucket_emit(g, s, slots, m, expected, col_base, c_col, c_val, err);
    return;
  }
  int64_t written = 0;
  for (int64_t r0 = 0; r0 < slots; r0 += g.size) {
    const int64_t slot = r0 + g.lane;
    int32_t k = kEmptyKey;
    double v = 0.0;
    if (slot < slots) {
      k = s.keys[slot];
      v = s.vals[slot];
    }
    const int64_t occ = (k != kEmptyKey) ? 1 : 0;
    int64_t total;
    const int64_t incl = group_scan<WARP>(g, occ, s.tmp, &total);
    g.sync();
    if (occ) {
      const int64_t pos = written + incl - 1;
      s.keys[pos] = k;
      s.vals[pos] = v;
    }
    written += total;
    g.sync();
  }
  int64_t P = 1;
  while (P < n) P <<= 1;
  if (P > slots) {  // only after a probe failure (table overfilled): give up on this row
    if (g.lane == 0) set_error(err, kErrHashFull);
    return;
  }
  for (int64_t j = n + g.lane; j < P; j += g.size) s.keys[j] = kPadKey;
  g.sync();
  for (int64_t kk = 2; kk <= P; kk <<= 1) {
    for (int64_t jj = kk >> 1; jj > 0; jj >>= 1) {
      for (int64_t i = g.lane; i < P; i += g.size) {
        const int64_t ixj = i ^ jj;
        if (ixj > i) {
          const int32_t ki = s.keys[i], kx = s.keys[ixj];
          const bool up = (i & kk) == 0;
          if ((ki > kx) == up) {
            s.keys[i] = kx;
            s.keys[ixj] = ki;
            const double t = s.vals[i];
            s.vals[i] = s.vals[ixj];
            s.vals[ixj] = t;
          }
        }
      }
      g.sync();
    }
  }
  if (n != expected && g.lane == 0) set_error(err, kErrRowOverflow);
  const int64_t m = n < expected ? n : expected;
  for (int64_t i = g.lane; i < m; i += g.size) {
    c_col[i] = s.keys[i] + col_base;
    c_val[i] = s.vals[i];
  }
}

// Ordered write of a dense accumulator: scan over the bitmap words.
template <bool WARP>
__device__ void dense_emit(const Group<WARP>& g, const Smem& s, int64_t width, int64_t expected,
                           int32_t col_base, int32_t* c_col, double* c_val, uint32_t* err) {
  const int64_t words = (width + 31) / 32;
  int64_t written = 0;
  for (int64_t w0 = 0; w0 < words; w0 += g.size) {
    const int64_t w = w0 + g.lane;
    const uint32_t bits = w < words ? static_cast<uint32_t>(s.keys[w]) : 0u;
    const int64_t c = __popc(bits);
    int64_t total;
    const int64_t incl = group_scan<WARP>(g, c, s.tmp, &total);
    int64_t pos = written + incl - c;
    uint32_t b = bits;
    while (b) {
      const int bit = __ffs(b) - 1;
      b &= b - 1;
      const int64_t idx = w * 32 + bit;
      if (pos < expected) {
        c_col[pos] = static_cast<int32_t>(idx) + col_base;
        c_val[pos] = s.vals[idx];
      }
      ++pos;
    }
    written += total;
  }
  if (written != expected && g.lane == 0) set_error(err, kErrRowOverflow);
}

// ---- the kernel --------------------------------------------------------------------------
template <bool WARP, bool NUMERIC, bool DENSE, bool CHUNK>
__global__ void __launch_bounds__(1024) k_accum(AccParams p) {
  extern __shared__ __align__(16) char smem_raw[];
  Group<WARP> g;
  int64_t item;
  char* region = smem_raw;
  const size_t gb = group_bytes(p.slots, WARP ? 32 : blockDim.x, DENSE, NUMERIC, !CHUNK);
  if (WARP) {
    const int w = threadIdx.x >> 5;
    g.lane = threadIdx.x & 31;
    g.size = 32;
    item = static_cast<int64_t>(blockIdx.x) * kWarpGroupsPerBlock + w;
    region += gb * w;
  } else {
    g.lane = threadIdx.x;
    g.size = blockDim.x;
    item = blockIdx.x;
  }
  if (item >= p.count) return;  // uniform per group
  const Smem s = carve(region, p.slots, g.size, DENSE, NUMERIC, !CHUNK);
  const uint32_t slots = static_cast<uint32_t>(p.slots);

  // identify the work item and its output
  int64_t grow;             // global row of C
  int32_t col_base = 0;     // column added on output
  int32_t acc_base = 0;     // dense accumulator origin (light dense rows)
  int64_t q = 0, cstart = 0, ccnt = 0;
  if (CHUNK) {
    q = p.list[item];
    cstart = p.cs.start[q];
    ccnt = p.cs.cnt[q];
    grow = p.cs.heavy_rows[p.cs.row[q]];
    col_base = p.cs.base[q];
  } else {
    grow = p.list[item];
    if (DENSE) acc_base = p.span_lo[grow];
  }
  const bool est = !CHUNK && NUMERIC && p.est_on;
  if (NUMERIC && !est && (grow < p.sink.row_begin || grow >= p.sink.row_end)) return;

  uint32_t* const flag = reinterpret_cast<uint32_t*>(s.tmp + 33);
  if (g.lane == 0) *flag = 0u;
  acc_clear<WARP, NUMERIC, DENSE>(g, s, p.slots);
  g.sync();
  int64_t fresh;
  if (CHUNK) fresh = expand_chunk<WARP, NUMERIC, DENSE>(g, s, p, cstart, ccnt, slots);
  else fresh = expand_row<WARP, NUMERIC, DENSE>(g, s, p, grow, acc_base, slots, est ? flag : p.err);
  g.sync();
  int64_t n;
  group_scan<WARP>(g, fresh, s.tmp, &n);
  if (!NUMERIC) {
    if (g.lane == 0) {
      if (CHUNK) p.cs.nnz[q] = n;
      else p.sink.row_nnz[grow] = n;
    }
    return;
  }
  if (est) {
    // estimated workflows: the row fits its capacity, or it is marked for the fallback pass
    g.sync();
    const bool over = *reinterpret_cast<volatile uint32_t*>(flag) != 0u || n > p.est.cap[grow];
    if (over) {
      if (g.lane == 0) p.est.est_nnz[grow] = -1;
      return;  // uniform per group
    }
    if (g.lane == 0) {
      p.est.est_nnz[grow] = n;
      p.sink.row_nnz[grow] = n;
    }
    const int64_t o = p.est.row_tmp[grow];
    if (DENSE) dense_emit<WARP>(g, s, p.slots, n, acc_base, p.est.tmp_col + o, p.est.tmp_val + o, p.err);
    else hash_emit<WARP>(g, s, p.slots, n, n, 0, p.est.tmp_col + o, p.est.tmp_val + o, p.err);
    return;
  }
  const int64_t rp0 = p.sink.row_ptr[grow];
  const int64_t win = p.sink.row_ptr[p.sink.row_begin];
  int64_t out, expected;
  if (CHUNK) {
    out = rp0 + p.cs.out[q] - win;
    expected = p.cs.nnz[q];  // counted by the symbolic phase
  } else {
    out = rp0 - win;
    expected = p.sink.row_ptr[grow + 1] - rp0;
  }
  g.sync();
  if (DENSE) {
    const int32_t base = CHUNK ? col_base : acc_base;
    dense_emit<WARP>(g, s, p.slots, expected, base, p.sink.c_col + out, p.sink.c_val + out, p.err);
  } else {
    hash_emit<WARP>(g, s, p.slots, n, expected, col_base, p.sink.c_col + out, p.sink.c_val + out,
                    p.err);
  }
}

size_t light_smem_bytes(int64_t slots, int tpr, bool dense, bool numeric) {
  const size_t gb = group_bytes(slots, tpr, dense, numeric, true);
  return tpr == 32 ? gb * kWarpGroupsPerBlock : gb;
}

template <bool WARP, bool NUMERIC, bool DENSE, bool CHUNK>
static void launch_one(const AccParams& p, int tpr, cudaStream_t s) {
  const size_t gb = group_bytes(p.slots, WARP ? 32 : tpr, DENSE, NUMERIC, !CHUNK);
  const size_t smem = WARP ? gb * kWarpGroupsPerBlock : gb;
  auto kern = k_accum<WARP, NUMERIC, DENSE, CHUNK>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  const int64_t blocks = WARP ? ceil_div(p.count, kWarpGroupsPerBlock) : p.count;
  const int threads = WARP ? 32 * kWarpGroupsPerBlock : tpr;
  note_launch();
  kern<<<static_cast<unsigned>(blocks), threads, smem, s>>>(p);
}

template <bool CHUNK>
static void dispatch(const AccParams& p, int tpr, bool dense, bool numeric, cudaStream_t s) {
  const bool warp = tpr == 32;
  if (warp) {
    if (numeric) {
      if (dense) launch_one<true, true, true, CHUNK>(p, tpr, s);
      else launch_one<true, true, false, CHUNK>(p, tpr, s);
    } else {
      if (dense) launch_one<true, false, true, CHUNK>(p, tpr, s);
      else launch_one<true, false, false, CHUNK>(p, tpr, s);
    }
  } else {
    if (numeric) {
      if (dense) launch_one<false, true, true, CHUNK>(p, tpr, s);
      else launch_one<false, true, false, CHUNK>(p, tpr, s);
    } else {
      if (dense) launch_one<false, false, true, CHUNK>(p, tpr, s);
      else launch_one<false, false, false, CHUNK>(p, tpr, s);
    }
  }
}

void launch_light(const spgemm_csr& A, const spgemm_csr& B, const int32_t* span_lo,
                  const RowJob& job, bool numeric, const Sink& sink, uint32_t* err,
                  cudaStream_t s, const EstSink* est) {
  if (job.count == 0) return;
  AccParams p{};
  if (est) {
    p.est = *est;
    p.est_on = 1;
  }
  p.arp = A.row_ptr;
  p.acol = A.col_idx;
  p.aval = A.vals;
  p.brp = B.row_ptr;
  p.bcol = B.col_idx;
  p.bval = B.vals;
  p.span_lo = span_lo;
  p.list = job.rows;
  p.count = job.count;
  p.slots = job.slots;
  p.sink = sink;
  p.err = err;
  p.has_vals = 1;
  dispatch<false>(p, job.tpr, job.dense, numeric, s);
}

void launch_chunks(const ChunkSet& cs, const int32_t* list, int64_t count, int64_t slots, int tpr,
                   bool dense, int64_t dense_width, bool numeric, const Sink& sink,
                   uint32_t* err, cudaStream_t s) {
  if (count == 0) return;
  AccParams p{};
  p.cs = cs;
  p.list = list;
  p.count = count;
  p.slots = dense ? dense_width : slots;
  p.sink = sink;
  p.err = err;
  p.has_vals = cs.val != nullptr;
  dispatch<true>(p, tpr, dense, numeric, s);
}

}  // namespace sg
