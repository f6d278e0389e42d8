// Shared-memory machinery of the chunk accumulators (gMAGNUS page, section III-E): a bitmap of
// the chunk's columns whose word prefix ranks every column (so the output needs no sort), the
// hash and dense value stores, and the hub-column copies of the dense accumulator.  Used by the
// accumulators that read C^_reord (k_chunk.cu) and by those that generate a chunk's products
// from A and the column-split B (k_fused.cu).
#pragma once

#include "internal.h"

namespace sg {

constexpr int kCkWarpsPerBlock = 8;

// Hub columns of a chunk: local columns with at most two set bits (0, 2^i, 2^i + 2^j) below
// 2^16.  In R-MAT / Kronecker power-law products the probability of a column falls with every
// set bit of its index, so these few columns take a large share of the products of every
// chunk (local column 0 alone ~2% on R-MAT with a = 0.57).  Shared-memory fp64 atomics
// serialise badly on one address, so hub products add into one of kHubCopies private copies of
// the hub slots (streaming warp w uses copy w mod kHubCopies); the copies are merged once per
// chunk.  Fewer copies contend, more copies lengthen the merge, a serial chain of fp64 adds per
// slot: with 1024-thread blocks 8 copies beat 31, 16 and 4; with the default 256-thread blocks
// 4 copies beat 8.  On other inputs the hubs are just ordinary columns.
constexpr int kHubCopies = 4;
constexpr int kHubBits = 16;
constexpr int kHubSlots = 1 + kHubBits + kHubBits * (kHubBits - 1) / 2;  // 137
static_assert(kHubSlots == kChunkHubSlots, "hub slot count");

// Branch-free (lanes of a warp that hit hubs and lanes that do not take the same path):
// 0 for column 0, 1 + i for 2^i, 1 + kHubBits + j(j-1)/2 + i for 2^i + 2^j (i < j), else -1.
__device__ __forceinline__ int hub_index(uint32_t c) {
  const int pc = __popc(c);
  const int i = __ffs(c) - 1;      // lowest set bit (-1 for c = 0)
  const int j = 31 - __clz(c);     // highest set bit
  const int two = 1 + kHubBits + ((j * (j - 1)) >> 1) + i;
  const int idx = pc == 0 ? 0 : (pc == 1 ? 1 + i : two);
  return (pc <= 2 && c < (1u << kHubBits)) ? idx : -1;
}

__host__ __device__ inline uint32_t hub_column(int idx) {
  if (idx == 0) return 0u;
  if (idx <= kHubBits) return 1u << (idx - 1);
  int k = idx - 1 - kHubBits, j = 1;
  while (k >= j) {
    k -= j;
    ++j;
  }
  return (1u << j) | (1u << k);
}

// Position of the k-th (0-based) set bit of m (k < popc(m)).
__device__ __forceinline__ int nth_set_bit(uint32_t m, int k) {
  int pos = 0;
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const uint32_t low = m & ((1u << w) - 1u);
    const int c = __popc(low);
    if (k >= c) {
      k -= c;
      m >>= w;
      pos += w;
    } else {
      m = low;
    }
  }
  return pos;
}

struct CkParams {
  ChunkSet cs;
  const int32_t* list;   // chunk ids of this bin
  int64_t count;
  int64_t width;         // bitmap width (columns of the widest chunk in the bin)
  int64_t slots;         // hash slots (hash numeric)
  Sink sink;
  uint32_t* err;
};

template <bool WARP>
struct CkGroup {
  int lane, size;
  __device__ __forceinline__ void sync() const {
    if (WARP) __syncwarp(); else __syncthreads();
  }
};

template <bool WARP>
__device__ __forceinline__ int64_t ck_scan(const CkGroup<WARP>& g, int64_t v, int64_t* tmp, int64_t* total) {
  if (WARP) {
    int64_t x = warp_incl_scan(v);
    *total = __shfl_sync(0xffffffffu, x, 31);
    return x;
  }
  return block_incl_scan(v, tmp, total);
}

__host__ __device__ inline size_t ck_align(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

// Shared memory of one group: scan scratch, bitmap words, prefix of the words, then the
// accumulator (hash keys + values, or dense values).
__host__ __device__ inline size_t ck_group_bytes(int64_t width, int64_t slots, int mode) {
  const int64_t words = (width + 31) / 32;
  size_t b = ck_align(33 * sizeof(int64_t)) + ck_align(words * 4) + ck_align(words * 4);
  if (mode == 1) b += ck_align(slots * 4) + ck_align(slots * 8);  // hash numeric
  if (mode == 2) b += ck_align(width * 8) + ck_align(kHubCopies * kHubSlots * 8);  // dense + hub copies
  if (mode == 3) b += ck_align(kHubCopies * kHubSlots * 8);                        // L2 dense: hubs only
  return b;
}

struct CkSmem {
  int64_t* tmp;
  uint32_t* bits;
  int32_t* pre;
  int32_t* keys;
  double* vals;
  double* hub;   // dense mode: private copies of the hub-column sums
};

__device__ __forceinline__ CkSmem ck_carve(char* p, int64_t width, int64_t slots, int mode) {
  const int64_t words = (width + 31) / 32;
  CkSmem s;
  s.tmp = reinterpret_cast<int64_t*>(p);
  p += ck_align(33 * sizeof(int64_t));
  s.bits = reinterpret_cast<uint32_t*>(p);
  p += ck_align(words * 4);
  s.pre = reinterpret_cast<int32_t*>(p);
  p += ck_align(words * 4);
  s.keys = nullptr;
  s.vals = nullptr;
  s.hub = nullptr;
  if (mode == 1) {
    s.keys = reinterpret_cast<int32_t*>(p);
    p += ck_align(slots * 4);
    s.vals = reinterpret_cast<double*>(p);
  } else if (mode == 2) {
    s.vals = reinterpret_cast<double*>(p);
    p += ck_align(width * 8);
    s.hub = reinterpret_cast<double*>(p);
  } else if (mode == 3) {
    s.hub = reinterpret_cast<double*>(p);
  }
  return s;
}

// Exclusive prefix of the bitmap word popcounts into s.pre; returns the number of set bits.
template <bool WARP>
__device__ __forceinline__ int64_t ck_bitmap_prefix(const CkGroup<WARP>& g, const CkSmem& s, int64_t words) {
  int64_t written = 0;
  for (int64_t w0 = 0; w0 < words; w0 += g.size) {
    const int64_t w = w0 + g.lane;
    const int64_t c = w < words ? __popc(s.bits[w]) : 0;
    int64_t tot;
    const int64_t incl = ck_scan<WARP>(g, c, s.tmp, &tot);
    if (w < words) s.pre[w] = static_cast<int32_t>(written + incl - c);
    written += tot;
  }
  return written;
}

__device__ __forceinline__ int32_t ck_rank(const CkSmem& s, int32_t col) {
  const uint32_t w = s.bits[col >> 5];
  return s.pre[col >> 5] + __popc(w & ((1u << (col & 31)) - 1u));
}


// Fold the hub copies into the dense value array (one thread per hub slot), then the ordered
// write of a dense chunk, balanced over the block: thread t writes output positions t, t + size,
// ... (consecutive threads, consecutive positions), finding its column by a binary search of the
// word prefix and a select inside the word (the bits of power-law inputs crowd into the low
// columns, so one thread per word would serialise the densest words).  The array is left zeroed
// and the bitmap cleared.  Every thread of the block calls it.
template <bool L2>
__device__ __forceinline__ void dense_fold_and_emit(const CkGroup<false>& g, const CkSmem& s, double* acc,
                                                    int64_t width, int64_t expected, int32_t base, int32_t* c_col,
                                                    double* c_val, uint32_t* err) {
  const int64_t words = (width + 31) / 32;
  for (int j = g.lane; j < kHubSlots; j += g.size) {
    const uint32_t c = hub_column(j);
    double sum = 0.0;
    for (int w = 0; w < kHubCopies; ++w) {
      sum += s.hub[w * kHubSlots + j];
      s.hub[w * kHubSlots + j] = 0.0;
    }
    if (c < width && sum != 0.0) {
      if (L2) __stcg(&acc[c], __ldcg(&acc[c]) + sum); else acc[c] += sum;
    }
  }
  if (L2) __threadfence_block();
  __syncthreads();
  const int64_t total = ck_bitmap_prefix(g, s, words);
  __syncthreads();
  if (total != expected && g.lane == 0) set_error(err, kErrRowOverflow);
  const int64_t n_out = total < expected ? total : expected;
  // four output positions per thread per step, their binary searches (last word whose prefix
  // is <= k: it holds bit number k) run in lockstep so the shared loads overlap
  int steps = 0;
  while ((int64_t(1) << steps) < words) ++steps;
  const int nw = static_cast<int>(words);
  for (int k0 = g.lane; k0 < static_cast<int>(total); k0 += 4 * g.size) {
    int lo[4], hi[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      lo[u] = 0;
      hi[u] = k0 + u * g.size < static_cast<int>(total) ? nw - 1 : 0;
    }
    for (int st = 0; st < steps; ++st) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (lo[u] < hi[u]) {
          const int mid = (lo[u] + hi[u] + 1) >> 1;
          if (s.pre[mid] <= k0 + u * g.size) lo[u] = mid; else hi[u] = mid - 1;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = k0 + u * g.size;
      if (k >= static_cast<int>(total)) continue;
      const int32_t idx = lo[u] * 32 + nth_set_bit(s.bits[lo[u]], k - s.pre[lo[u]]);
      if (k < n_out) {
        c_col[k] = idx + base;
        c_val[k] = L2 ? __ldcg(&acc[idx]) : acc[idx];
      }
      if (L2) __stcg(&acc[idx], 0.0); else acc[idx] = 0.0;  // leave the array zeroed
    }
  }
  __syncthreads();
  for (int64_t w = g.lane; w < words; w += g.size) s.bits[w] = 0u;
}

// Hash numeric finish: rank every occupied slot's column through the bitmap and write the
// chunk's entries at their final positions.  Every thread of the group calls it.
template <bool WARP>
__device__ __forceinline__ void hash_emit(const CkGroup<WARP>& g, const CkSmem& s, int64_t words, uint32_t slots,
                                          int64_t expected, int32_t base, int32_t* c_col, double* c_val,
                                          uint32_t* err) {
  const int64_t n = ck_bitmap_prefix<WARP>(g, s, words);
  g.sync();
  if (n != expected) {
    if (g.lane == 0) set_error(err, kErrRowOverflow);
    return;
  }
  for (uint32_t j = g.lane; j < slots; j += g.size) {
    const int32_t k = s.keys[j];
    if (k != kEmptyKey) {
      const int32_t r = ck_rank(s, k);
      c_col[r] = k + base;
      c_val[r] = s.vals[j];
    }
  }
}

// Insert one (column, value) product into the chunk's hash table (linear probing, columns as
// keys, values summed with shared atomics) and its bitmap.
__device__ __forceinline__ void hash_insert(const CkSmem& s, uint32_t slots, int32_t c, double v, uint32_t* err) {
  atomicOr(&s.bits[c >> 5], 1u << (c & 31));
  uint32_t slot = hash_slot(c, slots);
  uint32_t probe = 0;
  for (; probe < slots; ++probe) {
    const int32_t k = *reinterpret_cast<volatile int32_t*>(&s.keys[slot]);
    if (k == c) break;
    if (k == kEmptyKey) {
      const int32_t old = atomicCAS(&s.keys[slot], kEmptyKey, c);
      if (old == kEmptyKey || old == c) break;
    }
    slot = (slot + 1 == slots) ? 0 : slot + 1;
  }
  if (probe < slots) atomicAdd(&s.vals[slot], v);
  else set_error(err, kErrHashFull);
}

}  // namespace sg
