// Accumulation of the final chunks of C^_reord (gMAGNUS page, section III-E), for chunks whose
// column width fits a shared-memory bitmap (every last-level chunk, width W).
//
//   symbolic : one bit per column of the chunk; the chunk's nnz is the number of set bits.
//   numeric  : small chunks sum in a hash map (load factor <= 1/2); large chunks sum in a dense
//              array of W doubles whose slots are zeroed on first touch (the bitmap tells which
//              slots are live, so the array is never cleared as a whole).  In both cases the
//              output order comes from the bitmap: the rank of column c inside the chunk is the
//              number of set bits below c (a block scan over the bitmap words), so no sort is
//              needed, and each entry is written straight to its final position in C.
#include "internal.h"

namespace sg {

constexpr int kCkWarpsPerBlock = 8;

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
  if (mode == 2) b += ck_align(width * 8);                          // dense numeric
  return b;
}

struct CkSmem {
  int64_t* tmp;
  uint32_t* bits;
  int32_t* pre;
  int32_t* keys;
  double* vals;
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
  if (mode == 1) {
    s.keys = reinterpret_cast<int32_t*>(p);
    p += ck_align(slots * 4);
    s.vals = reinterpret_cast<double*>(p);
  } else if (mode == 2) {
    s.vals = reinterpret_cast<double*>(p);
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

// mode 0: symbolic, 1: hash numeric, 2: dense numeric
template <bool WARP, int MODE>
__global__ void __launch_bounds__(1024) k_chunk(CkParams p) {
  extern __shared__ __align__(16) char smem_raw[];
  CkGroup<WARP> g;
  int64_t item;
  char* region = smem_raw;
  const size_t gb = ck_group_bytes(p.width, p.slots, MODE);
  if (WARP) {
    const int w = threadIdx.x >> 5;
    g.lane = threadIdx.x & 31;
    g.size = 32;
    item = static_cast<int64_t>(blockIdx.x) * kCkWarpsPerBlock + w;
    region += gb * w;
  } else {
    g.lane = threadIdx.x;
    g.size = blockDim.x;
    item = blockIdx.x;
  }
  if (item >= p.count) return;
  const CkSmem s = ck_carve(region, p.width, p.slots, MODE);
  const int64_t q = p.list[item];
  const int64_t start = p.cs.start[q];
  const int64_t cnt = p.cs.cnt[q];
  const int64_t grow = p.cs.heavy_rows[p.cs.row[q]];
  if (MODE != 0 && (grow < p.sink.row_begin || grow >= p.sink.row_end)) return;
  const int64_t words = (p.width + 31) / 32;
  const uint32_t width = static_cast<uint32_t>(p.width);
  const uint32_t slots = static_cast<uint32_t>(p.slots);
  for (int64_t w = g.lane; w < words; w += g.size) s.bits[w] = 0u;
  if (MODE == 1)
    for (int64_t j = g.lane; j < p.slots; j += g.size) s.keys[j] = kEmptyKey;
  if (MODE != 1) g.sync();
  const int32_t* col = p.cs.col + start;
  const double* val = p.cs.val + start;

  if (MODE == 0) {
    for (int64_t f = g.lane; f < cnt; f += g.size) {
      const uint32_t c = static_cast<uint32_t>(col[f]);
      if (c < width) atomicOr(&s.bits[c >> 5], 1u << (c & 31));
      else set_error(p.err, kErrBounds);
    }
    g.sync();
    int64_t n = 0;
    for (int64_t w = g.lane; w < words; w += g.size) n += __popc(s.bits[w]);
    int64_t tot;
    ck_scan<WARP>(g, n, s.tmp, &tot);
    if (g.lane == 0) p.cs.nnz[q] = tot;
    return;
  }

  const int64_t rp0 = p.sink.row_ptr[grow];
  const int64_t out = rp0 + p.cs.out[q] - p.sink.row_ptr[p.sink.row_begin];
  const int64_t expected = p.cs.nnz[q];
  int32_t* c_col = p.sink.c_col + out;
  double* c_val = p.sink.c_val + out;
  const int32_t base = p.cs.base[q];

  if (MODE == 1) {
    // keys and values were cleared above (values here, keys with the bitmap)
    for (int64_t j = g.lane; j < p.slots; j += g.size) s.vals[j] = 0.0;
    g.sync();
    for (int64_t f = g.lane; f < cnt; f += g.size) {
      const int32_t c = col[f];
      if (static_cast<uint32_t>(c) >= width) {
        set_error(p.err, kErrBounds);
        continue;
      }
      const double v = val[f];
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
      else set_error(p.err, kErrHashFull);
    }
    g.sync();
    const int64_t n = ck_bitmap_prefix<WARP>(g, s, words);
    g.sync();
    if (n != expected) {
      if (g.lane == 0) set_error(p.err, kErrRowOverflow);
      return;
    }
    for (int64_t j = g.lane; j < p.slots; j += g.size) {
      const int32_t k = s.keys[j];
      if (k != kEmptyKey) {
        const int32_t r = ck_rank(s, k);
        c_col[r] = k + base;
        c_val[r] = s.vals[j];
      }
    }
    return;
  }

  if (MODE == 2) {
    // dense: a value slot is zeroed by the thread whose atomicOr first sets its bit; adds
    // follow after a barrier, so no add can meet an unzeroed slot
    constexpr int kItems = 4;
    for (int64_t b0 = 0; b0 < cnt; b0 += static_cast<int64_t>(g.size) * kItems) {
      int32_t cr[kItems];
      double vr[kItems];
#pragma unroll
      for (int j = 0; j < kItems; ++j) {
        const int64_t f = b0 + static_cast<int64_t>(j) * g.size + g.lane;
        cr[j] = -1;
        vr[j] = 0.0;
        if (f < cnt) {
          const int32_t c = col[f];
          if (static_cast<uint32_t>(c) < width) {
            cr[j] = c;
            vr[j] = val[f];
            const uint32_t bit = 1u << (c & 31);
            const uint32_t old = atomicOr(&s.bits[c >> 5], bit);
            if (!(old & bit)) s.vals[c] = 0.0;
          } else {
            set_error(p.err, kErrBounds);
          }
        }
      }
      g.sync();
#pragma unroll
      for (int j = 0; j < kItems; ++j)
        if (cr[j] >= 0) atomicAdd(&s.vals[cr[j]], vr[j]);
    }
    g.sync();
    // ordered output: scan of the bitmap words, then every word writes its set bits
    int64_t written = 0;
    for (int64_t w0 = 0; w0 < words; w0 += g.size) {
      const int64_t w = w0 + g.lane;
      const uint32_t bits = w < words ? s.bits[w] : 0u;
      const int64_t c = __popc(bits);
      int64_t tot;
      const int64_t incl = ck_scan<WARP>(g, c, s.tmp, &tot);
      int64_t pos = written + incl - c;
      uint32_t b = bits;
      while (b) {
        const int bit = __ffs(b) - 1;
        b &= b - 1;
        const int32_t idx = static_cast<int32_t>(w * 32 + bit);
        if (pos < expected) {
          c_col[pos] = idx + base;
          c_val[pos] = s.vals[idx];
        }
        ++pos;
      }
      written += tot;
    }
    if (written != expected && g.lane == 0) set_error(p.err, kErrRowOverflow);
  }
}

size_t chunk_smem_bytes(int64_t width, int64_t slots, int mode, bool warp) {
  const size_t gb = ck_group_bytes(width, slots, mode);
  return warp ? gb * kCkWarpsPerBlock : gb;
}

template <bool WARP, int MODE>
static void ck_launch(const CkParams& p, int tpr, cudaStream_t s) {
  const size_t smem = chunk_smem_bytes(p.width, p.slots, MODE, WARP);
  auto kern = k_chunk<WARP, MODE>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  const int64_t blocks = WARP ? ceil_div(p.count, kCkWarpsPerBlock) : p.count;
  const int threads = WARP ? 32 * kCkWarpsPerBlock : tpr;
  note_launch();
  kern<<<static_cast<unsigned>(blocks), threads, smem, s>>>(p);
}

void launch_chunk_bitmap(const ChunkSet& cs, const int32_t* list, int64_t count, int64_t width, int mode,
                         int64_t slots, int tpr, const Sink& sink, uint32_t* err, cudaStream_t s) {
  if (count == 0) return;
  CkParams p{};
  p.cs = cs;
  p.list = list;
  p.count = count;
  p.width = width;
  p.slots = slots;
  p.sink = sink;
  p.err = err;
  const bool warp = tpr == 32;
  if (mode == 0) {
    if (warp) ck_launch<true, 0>(p, tpr, s); else ck_launch<false, 0>(p, tpr, s);
  } else if (mode == 1) {
    if (warp) ck_launch<true, 1>(p, tpr, s); else ck_launch<false, 1>(p, tpr, s);
  } else {
    ck_launch<false, 2>(p, tpr, s);
  }
}

}  // namespace sg
