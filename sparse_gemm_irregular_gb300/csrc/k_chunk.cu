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
#include <algorithm>

#include "chunk_common.cuh"

namespace sg {

// mode 0: symbolic, 1: hash numeric (the dense numeric accumulator is k_chunk_dense below)
// Warp groups launch 8 warps per block, block groups at most 512 threads (kChunkTpr).
template <bool WARP, int MODE>
__global__ void __launch_bounds__(WARP ? 32 * kCkWarpsPerBlock : 512) k_chunk(CkParams p) {
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
  // hash numeric in blocks: the table is sized for this chunk (a power of two >= 2 x its
  // elements, at most the bin's slots), so clearing and scanning it cost in proportion to the
  // chunk (4.86 -> 4.56 ms on R-MAT s18; warps keep their full 512-slot tables, where the
  // smaller ones measured slower)
  uint32_t slots = static_cast<uint32_t>(p.slots);
  if (MODE == 1 && !WARP) {
    uint32_t need = 64;
    while (need < 2 * cnt && need < slots) need <<= 1;
    slots = need < slots ? need : slots;
  }
  for (int64_t w = g.lane; w < words; w += g.size) s.bits[w] = 0u;
  if (MODE == 1)
    for (uint32_t j = g.lane; j < slots; j += g.size) s.keys[j] = kEmptyKey;
  if (MODE != 1) g.sync();
  const int32_t* col = p.cs.col + start;
  const double* val = p.cs.val + start;
  // element offsets inside a chunk are 32-bit (a chunk of 2^31 or more elements is rejected)
  if (cnt > 0x7fffffffLL) {
    if (g.lane == 0) set_error(p.err, kErrBounds);
    return;
  }
  const int n32 = static_cast<int>(cnt);

  if (MODE == 0) {
    constexpr int U = 8;
    for (int f0 = 0; f0 < n32; f0 += g.size * U) {
      uint32_t cr[U];
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int f = f0 + j * g.size + g.lane;
        cr[j] = f < n32 ? static_cast<uint32_t>(__ldcs(col + f)) : 0xffffffffu;
      }
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const uint32_t c = cr[j];
        if (c < width) atomicOr(&s.bits[c >> 5], 1u << (c & 31));
        else if (c != 0xffffffffu) set_error(p.err, kErrBounds);
      }
    }
    g.sync();
    int64_t n = 0;
    for (int w = g.lane; w < static_cast<int>(words); w += g.size) n += __popc(s.bits[w]);
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
    for (uint32_t j = g.lane; j < slots; j += g.size) s.vals[j] = 0.0;
    g.sync();
    constexpr int U = 4;
    for (int f0 = 0; f0 < n32; f0 += g.size * U) {
      int32_t cr[U];
      double vr[U];
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int f = f0 + j * g.size + g.lane;
        cr[j] = -1;
        vr[j] = 0.0;
        if (f < n32) {
          cr[j] = __ldcs(col + f);
          vr[j] = __ldcs(val + f);
        }
      }
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int32_t c = cr[j];
        if (c < 0) continue;
        if (static_cast<uint32_t>(c) >= width) {
          set_error(p.err, kErrBounds);
          continue;
        }
        hash_insert(s, slots, c, vr[j], p.err);
      }
    }
    g.sync();
    hash_emit<WARP>(g, s, words, slots, expected, base, c_col, c_val, p.err);
  }
}

// Dense numeric accumulation as persistent blocks (as many per SM as the W-double value arrays
// allow: three 256-thread blocks at the default W = 8192).  With few blocks per SM the per-chunk latency (taking the next
// chunk from the work counter, the chain of descriptor loads) would sit on the critical path, so
// warp 0 is a helper: while the other warps stream the current chunk it takes the next chunk and
// loads its descriptor into a second shared slot.  The value array is zeroed once and every
// chunk clears the slots it writes.  Hub columns (hub_index) add into private copies of their
// sums in shared memory, merged once per chunk, so the hottest columns of power-law inputs do
// not serialise on one address.  The L2 variant keeps the value array in an L2-resident global
// slice instead (fire-and-forget reductions), for A/B measurements.
struct DenseJob {
  int64_t start, cnt, out, expected;
  int32_t base;
  int32_t state;  // 0 none left, 1 work, 2 outside the numeric row window
};

__device__ __forceinline__ void dense_fetch(const CkParams& p, int* next, DenseJob* j) {
  const int64_t item = atomicAdd(next, 1);
  if (item >= p.count) {
    j->state = 0;
    return;
  }
  const int64_t q = p.list[item];
  const int64_t grow = p.cs.heavy_rows[p.cs.row[q]];
  if (grow < p.sink.row_begin || grow >= p.sink.row_end) {
    j->state = 2;
    return;
  }
  j->start = p.cs.start[q];
  j->cnt = p.cs.cnt[q];
  if (j->cnt > 0x7fffffffLL) {  // element offsets inside a chunk are 32-bit
    set_error(p.err, kErrBounds);
    j->state = 2;
    return;
  }
  j->out = p.sink.row_ptr[grow] + p.cs.out[q] - p.sink.row_ptr[p.sink.row_begin];
  j->expected = p.cs.nnz[q];
  j->base = p.cs.base[q];
  j->state = 1;
}

// One instantiation per block size, with the register budget of three blocks per SM (the default
// W = 8192 fits three value arrays per SM) or of one 1024-thread block.
template <bool L2, int THREADS>
__global__ void __launch_bounds__(THREADS, THREADS == 256 ? 3 : (THREADS == 512 ? 2 : 1))
    k_chunk_dense(CkParams p, int* next, double* gacc_all) {
  extern __shared__ __align__(16) char smem_raw[];
  __shared__ DenseJob jobs[3];  // current, next, and the one the helper is fetching
  CkGroup<false> g;
  g.lane = threadIdx.x;
  g.size = blockDim.x;
  const CkSmem s = ck_carve(smem_raw, p.width, 0, L2 ? 3 : 2);
  const int64_t words = (p.width + 31) / 32;
  const uint32_t width = static_cast<uint32_t>(p.width);
  const int warp = threadIdx.x >> 5;
  const int nwork = (blockDim.x >> 5) - 1;  // streaming warps 1..nwork
  const int nt = nwork * 32;
  const int t = static_cast<int>(threadIdx.x) - 32;
  double* acc = L2 ? gacc_all + static_cast<int64_t>(blockIdx.x) * p.width : s.vals;
  double* my_hub = s.hub + ((warp > 0 ? warp - 1 : 0) % kHubCopies) * kHubSlots;
  if (L2) {
    for (int64_t j = g.lane; j < p.width; j += g.size) __stcg(&acc[j], 0.0);
  } else {
    double2* v2 = reinterpret_cast<double2*>(acc);
    for (int64_t j = g.lane; j < p.width / 2; j += g.size) v2[j] = make_double2(0.0, 0.0);
    if ((p.width & 1) && g.lane == 0) acc[p.width - 1] = 0.0;
  }
  for (int j = g.lane; j < kHubCopies * kHubSlots; j += g.size) s.hub[j] = 0.0;
  for (int64_t w = g.lane; w < words; w += g.size) s.bits[w] = 0u;
  if (threadIdx.x == 0) {
    dense_fetch(p, next, &jobs[0]);
    if (jobs[0].state != 0) dense_fetch(p, next, &jobs[1]);
    else jobs[1].state = 0;
  }
  __syncthreads();
  // streaming registers: batch b of the current chunk is loaded while batch b-1 is added.  A
  // chunk is a base pointer pair and a 32-bit count held in registers, so the per-element work
  // is 32-bit offset arithmetic (no rereads of the shared descriptors).
  constexpr int U = 4;
  int32_t cr[U];
  double vr[U];
  auto load_batch = [&](const int32_t* bc, const double* bv, int n, int f0) {
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int f = f0 + j * nt + t;
      cr[j] = -1;
      if (f < n) {
        cr[j] = __ldcs(bc + f);
        vr[j] = __ldcs(bv + f);
      }
    }
  };
  auto chunk_of = [&](const DenseJob& jb, const int32_t*& bc, const double*& bv, int& n) {
    n = jb.state == 1 ? static_cast<int>(jb.cnt) : 0;
    bc = p.cs.col + (jb.state == 1 ? jb.start : 0);
    bv = p.cs.val + (jb.state == 1 ? jb.start : 0);
  };
  const int32_t* ccol;
  const double* cval;
  int ccnt;
  chunk_of(jobs[0], ccol, cval, ccnt);
  if (warp > 0) load_batch(ccol, cval, ccnt, 0);
  for (int it = 0;; ++it) {
    const DenseJob job = jobs[it % 3];
    if (job.state == 0) break;
    if (warp == 0) {
      if (threadIdx.x == 0) {
        const DenseJob nx = jobs[(it + 1) % 3];
        if (nx.state != 0) dense_fetch(p, next, &jobs[(it + 2) % 3]);
        else jobs[(it + 2) % 3].state = 0;
      }
    } else {
      const int32_t* ncol;
      const double* nval;
      int ncnt;
      chunk_of(jobs[(it + 1) % 3], ncol, nval, ncnt);
      const int step = nt * U;
      for (int f0 = 0; f0 < (ccnt > 0 ? ccnt : 1); f0 += step) {
        int32_t c2[U];
        double v2[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
          c2[j] = cr[j];
          v2[j] = vr[j];
        }
        // next batch of this chunk, or the first batch of the next chunk
        if (f0 + step < ccnt) load_batch(ccol, cval, ccnt, f0 + step);
        else load_batch(ncol, nval, ncnt, 0);
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const int32_t c = c2[j];
          if (c < 0) continue;
          if (static_cast<uint32_t>(c) < width) {
            atomicOr(&s.bits[c >> 5], 1u << (c & 31));
            const int hi = hub_index(static_cast<uint32_t>(c));
            if (L2) {
              if (hi >= 0) atomicAdd(&my_hub[hi], v2[j]);
              else atomicAdd(&acc[c], v2[j]);
            } else {
              atomicAdd(hi >= 0 ? &my_hub[hi] : &acc[c], v2[j]);  // one shared atomic, address selected
            }
          } else {
            set_error(p.err, kErrBounds);
          }
        }
      }
      ccol = ncol;
      cval = nval;
      ccnt = ncnt;
    }
    if (L2) __threadfence_block();
    __syncthreads();
    if (job.state == 1)
      dense_fold_and_emit<L2>(g, s, acc, p.width, job.expected, job.base, p.sink.c_col + job.out,
                              p.sink.c_val + job.out, p.err);
    __syncthreads();
  }
}

// ---- the hash bins as persistent groups ---------------------------------------------------
// Chunks of at most 1024 elements are the most numerous (R-MAT scale 21: 1.6e8 of them, 68 and
// 522 elements on average in the two bins), so the work that does not scale with the elements
// decides their cost.  A group (a warp for chunks of at most kWarpChunkMax elements, a 128-thread
// block for the rest) keeps its shared table across chunks and takes chunk i, i + (groups of the
// grid), ...:
//   - the chunk's descriptor comes from a prepass (one 32-byte load, issued a chunk ahead);
//   - the hash table is the smallest power of two >= 2 x elements (at least 64 slots), so the
//     final sweep is proportional to the chunk;
//   - the bitmap prefix is one warp scan: lane l sums its run of consecutive words;
//   - the final sweep writes every occupied slot at its rank and empties the slots it visits,
//     and the group zeroes the bitmap words, so no chunk clears the whole table.
template <int T>
struct GroupCfg {
  static constexpr int kMax = T == 32 ? static_cast<int>(kWarpChunkMax) : static_cast<int>(kBlockChunkMax);
  static constexpr int kSlots = 2 * kMax;
  static constexpr int kBlock = T == 32 ? 256 : T;   // eight warp groups per block, or one block group
  static constexpr int kGroups = kBlock / T;
  static constexpr int kPerThread = kMax / T;        // elements per thread of the largest chunk
};

__global__ void k_chunk_desc(ChunkSet cs, const int32_t* __restrict__ list, int64_t count, int64_t max_cnt, Sink sink,
                             ChunkDesc* __restrict__ desc, uint32_t* err) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= count) return;
  const int64_t q = list[i];
  const int64_t grow = cs.heavy_rows[cs.row[q]];
  ChunkDesc d{};
  d.cnt = -1;
  const int64_t cnt = cs.cnt[q];
  if (grow >= sink.row_begin && grow < sink.row_end) {
    if (cnt > max_cnt) {
      set_error(err, kErrBounds);
    } else {
      d.start = cs.start[q];
      d.out = sink.row_ptr[grow] + cs.out[q] - sink.row_ptr[sink.row_begin];
      d.cnt = static_cast<int32_t>(cnt);
      d.expected = static_cast<int32_t>(cs.nnz[q]);
      d.base = cs.base[q];
    }
  }
  desc[i] = d;
}

// bitmap words per lane of the prefix warp (a multiple of 4, so that a lane's run is whole uint4s)
__host__ __device__ inline int64_t grp_words_per_lane(int64_t width) {
  const int64_t p = ((width + 31) / 32 + 31) / 32;
  return (p + 3) & ~int64_t(3);
}

template <int T>
__host__ __device__ inline size_t grp_bytes(int64_t width) {
  const int64_t words = 32 * grp_words_per_lane(width);  // bitmap and prefix, padded to whole lane runs
  return ck_align(words * 4) * 2 + ck_align(GroupCfg<T>::kSlots * 4) + ck_align(GroupCfg<T>::kSlots * 8) + 16;
}

template <int T>
__device__ __forceinline__ void grp_sync() {
  if (T == 32) __syncwarp(); else __syncthreads();
}

template <int T>
__global__ void __launch_bounds__(GroupCfg<T>::kBlock) k_chunk_groups(ChunkSet cs, const ChunkDesc* __restrict__ desc,
                                                                    int64_t count, int64_t width, Sink sink,
                                                                    uint32_t* err) {
  using C = GroupCfg<T>;
  extern __shared__ __align__(16) char smem_raw[];
  const int gi = threadIdx.x / T;
  const int t = threadIdx.x % T;
  const int lane = threadIdx.x & 31;
  const int P = static_cast<int>(grp_words_per_lane(width));
  const int nwords = 32 * P;
  char* region = smem_raw + grp_bytes<T>(width) * gi;
  uint32_t* bits = reinterpret_cast<uint32_t*>(region);
  int32_t* pre = reinterpret_cast<int32_t*>(region + ck_align(nwords * 4));
  int32_t* keys = reinterpret_cast<int32_t*>(region + 2 * ck_align(nwords * 4));
  double* vals = reinterpret_cast<double*>(region + 2 * ck_align(nwords * 4) + ck_align(C::kSlots * 4));
  int32_t* tot = reinterpret_cast<int32_t*>(region + 2 * ck_align(nwords * 4) + ck_align(C::kSlots * 4) +
                                            ck_align(C::kSlots * 8));
  for (int j = t; j < nwords; j += T) bits[j] = 0u;
  for (int j = t; j < C::kSlots; j += T) {
    keys[j] = kEmptyKey;
    vals[j] = 0.0;
  }
  grp_sync<T>();
  CkSmem s{};
  s.bits = bits;
  s.pre = pre;
  s.keys = keys;
  s.vals = vals;
  const uint32_t uw = static_cast<uint32_t>(width);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * C::kGroups;
  int64_t item = static_cast<int64_t>(blockIdx.x) * C::kGroups + gi;
  ChunkDesc d{};
  d.cnt = -1;
  if (item < count) d = desc[item];
  while (item < count) {
    const int64_t nitem = item + stride;
    ChunkDesc nd{};
    nd.cnt = -1;
    if (nitem < count) nd = desc[nitem];  // in flight while this chunk is summed
    const int n = d.cnt;
    if (n > 0) {
      uint32_t S = 64;
      while (S < 2u * static_cast<uint32_t>(n) && S < static_cast<uint32_t>(C::kSlots)) S <<= 1;
      const int32_t* col = cs.col + d.start;
      const double* val = cs.val + d.start;
      int32_t cr[C::kPerThread];
      double vr[C::kPerThread];
#pragma unroll
      for (int j = 0; j < C::kPerThread; ++j) {
        const int f = j * T + t;
        cr[j] = -1;
        vr[j] = 0.0;
        if (f < n) {
          cr[j] = __ldcs(col + f);
          vr[j] = __ldcs(val + f);
        }
      }
#pragma unroll
      for (int j = 0; j < C::kPerThread; ++j) {
        const int32_t c = cr[j];
        if (c < 0) continue;
        if (static_cast<uint32_t>(c) >= uw) {
          set_error(err, kErrBounds);
          continue;
        }
        hash_insert(s, S, c, vr[j], err);
      }
      grp_sync<T>();
      // rank of every bitmap word, by the group's first warp: lane l owns words [l P, l P + P)
      if (t < 32) {
        const uint4* b4 = reinterpret_cast<const uint4*>(bits + lane * P);
        int32_t run = 0;
        for (int j = 0; j < P / 4; ++j) {
          const uint4 x = b4[j];
          run += __popc(x.x) + __popc(x.y) + __popc(x.z) + __popc(x.w);
        }
        const int32_t incl = warp_incl_scan(run);
        int32_t acc = incl - run;
        int4* p4 = reinterpret_cast<int4*>(pre + lane * P);
        for (int j = 0; j < P / 4; ++j) {
          const uint4 x = b4[j];
          int4 o;
          o.x = acc;
          o.y = o.x + __popc(x.x);
          o.z = o.y + __popc(x.y);
          o.w = o.z + __popc(x.z);
          acc = o.w + __popc(x.w);
          p4[j] = o;
        }
        if (lane == 31) *tot = incl;
      }
      grp_sync<T>();
      const bool ok = *tot == d.expected;
      if (!ok && t == 0) set_error(err, kErrRowOverflow);
      int32_t* c_col = sink.c_col + d.out;
      double* c_val = sink.c_val + d.out;
      for (uint32_t j = t; j < S; j += T) {
        const int32_t k = keys[j];
        if (k != kEmptyKey) {
          if (ok) {
            const int32_t r = ck_rank(s, k);
            c_col[r] = k + d.base;
            c_val[r] = vals[j];
          }
          keys[j] = kEmptyKey;
          vals[j] = 0.0;
        }
      }
      grp_sync<T>();
      uint4* z4 = reinterpret_cast<uint4*>(bits);
      for (int j = t; j < nwords / 4; j += T) z4[j] = make_uint4(0u, 0u, 0u, 0u);
      grp_sync<T>();
    }
    d = nd;
    item = nitem;
  }
}

template <int T>
static void groups_launch(const ChunkSet& cs, const ChunkDesc* desc, int64_t count, int64_t width, const Sink& sink,
                          uint32_t* err, int sms, cudaStream_t s) {
  using C = GroupCfg<T>;
  const size_t smem = grp_bytes<T>(width) * C::kGroups;
  cudaFuncSetAttribute(k_chunk_groups<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_chunk_groups<T>, C::kBlock, smem);
  if (per_sm < 1) per_sm = 1;
  const int64_t blocks = std::min<int64_t>(ceil_div(count, C::kGroups), static_cast<int64_t>(sms) * per_sm);
  note_launch();
  k_chunk_groups<T><<<static_cast<unsigned>(blocks), C::kBlock, smem, s>>>(cs, desc, count, width, sink, err);
}

void launch_chunk_groups(const ChunkSet& cs, const int32_t* list, int64_t count, int64_t width, bool warps,
                         const Sink& sink, ChunkDesc* desc, uint32_t* err, cudaStream_t s) {
  if (count == 0) return;
  note_launch();
  k_chunk_desc<<<static_cast<unsigned>(ceil_div(count, 256)), 256, 0, s>>>(
      cs, list, count, warps ? kWarpChunkMax : kBlockChunkMax, sink, desc, err);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (warps) groups_launch<32>(cs, desc, count, width, sink, err, sms, s);
  else groups_launch<128>(cs, desc, count, width, sink, err, sms, s);
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
                         int64_t slots, int tpr, const Sink& sink, uint32_t* err, int* counter, double* gacc,
                         cudaStream_t s) {
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
    int dev = 0, sms = 0, smem_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaMemsetAsync(counter, 0, sizeof(int), s);
    note_launch();
    if (gacc) {  // L2-resident accumulators (one per SM): the shared array is not needed
      const int64_t blocks = std::min<int64_t>(count, sms);
      const size_t smem = chunk_smem_bytes(width, 0, 3, false);
      cudaFuncSetAttribute(k_chunk_dense<true, 1024>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
      k_chunk_dense<true, 1024><<<static_cast<unsigned>(blocks), 1024, smem, s>>>(p, counter, gacc);
    } else {
      // as many blocks per SM as the value arrays allow; the block shrinks with them (three
      // 256-thread blocks of W = 8192 beat two of 512 threads and one of 1024 at W = 16384)
      const size_t smem = chunk_smem_bytes(width, 0, 2, false);
      const int fit = static_cast<int>(smem_sm / (smem + 1024));
      // (384-thread blocks at three per SM measured slower: 15.3 against 14.6 ms on R-MAT s18)
      const int threads = fit >= 3 ? 256 : (fit == 2 ? 512 : 1024);
      auto kern = threads == 256 ? k_chunk_dense<false, 256>
                                 : (threads == 512 ? k_chunk_dense<false, 512> : k_chunk_dense<false, 1024>);
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      int per_sm = 1;
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
      if (per_sm < 1) per_sm = 1;
      const int64_t blocks = std::min<int64_t>(count, static_cast<int64_t>(sms) * per_sm);
      kern<<<static_cast<unsigned>(blocks), threads, smem, s>>>(p, counter, nullptr);
    }
  }
}

}  // namespace sg
