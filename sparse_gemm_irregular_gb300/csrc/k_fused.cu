// Heavy rows without the intermediate matrix in HBM (SPGEMM_FLAG_FUSED).
//
// gMAGNUS (section III-A, Algorithm 3) expands the heavy rows into C^ with an outer product,
// then multisplits C^ by column range into C^_reord, whose rows (one per (heavy row, chunk))
// are accumulated in shared memory.  The chunk of a product A[r,k] * B[k,j] is j >> log2(W):
// it depends only on the column of the B entry.  So the multisplit can be applied once to the
// rows of B instead of to the products (O(nnz B) instead of O(IP)): every row k of B is split
// into its entries of chunk 0, chunk 1, ... (k_bsplit).  The products of C^_reord row (r, c)
// are then exactly { A[r,k] * B_split[k, chunk c] : k in row r of A }, and the chunk
// accumulator generates them itself, from A and the split B, instead of reading them from
// C^_reord.  C^ and C^_reord never reach HBM; the level-0 histogram (elements per (row,
// chunk)) is the factorised one of k_row_chunk_counts, and the final chunks, their bins, the
// bitmap-ordered output and the offsets inside the rows of C are those of the expanded path.
//
// Product generator (fused_products): one warp takes a window of 32 entries of row r of A;
// lane l reads, from the batch's segment table, the range (segment) of row k_l of B_split that
// lies in chunk c.  Segments of 16 or more products -- most of the products of power-law
// inputs, which come from the long rows of B -- are swept by the whole warp one at a time.  The
// short ones are flattened: a warp scan of their lengths, then in every round lane l takes
// product f0 + l, finding its entry by a five-step binary search over the lanes' inclusive sums
// (shuffles).  Either way consecutive lanes read consecutive entries of B_split.  The blocks of
// the larger chunks deal the rounds of products out over their warps.
#include <algorithm>

#include "chunk_common.cuh"

namespace sg {

// ---- the column split of B ---------------------------------------------------------------------
constexpr int kBsWarps = 4;   // rows of B per block (one warp each)

// Rows of B that some heavy row of A uses (colcnt[k] > 0): bo[k * (v + 1) + c] = offset of the
// row's chunk-c entries inside the row (exclusive prefix of bh[k * v + .], bo[.. + v] = row
// length), and the row's entries regrouped by chunk at the same row range of bs_col / bs_val.
// Order inside a chunk group is not kept (the accumulators sum in any order).
template <bool VALS>
__global__ void __launch_bounds__(32 * kBsWarps) k_bsplit(const int64_t* __restrict__ brp,
                                                        const int32_t* __restrict__ bcol,
                                                        const double* __restrict__ bval, int64_t krows,
                                                        const int32_t* __restrict__ colcnt,
                                                        const int32_t* __restrict__ bh, int shift, int64_t v,
                                                        int32_t* __restrict__ bo, int32_t* __restrict__ bs_col,
                                                        double* __restrict__ bs_val, uint32_t* err) {
  extern __shared__ int32_t bs_cursor[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t k = static_cast<int64_t>(blockIdx.x) * kBsWarps + warp;
  if (k >= krows || colcnt[k] == 0) return;
  int32_t* cur = bs_cursor + warp * v;
  int32_t* out = bo + k * (v + 1);
  int32_t run = 0;
  for (int64_t c0 = 0; c0 < v; c0 += 32) {
    const int64_t c = c0 + lane;
    const int32_t x = c < v ? bh[k * v + c] : 0;
    const int32_t incl = warp_incl_scan(x);
    if (c < v) {
      cur[c] = run + incl - x;
      out[c] = run + incl - x;
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) out[v] = run;
  __syncwarp();
  const int64_t b0 = brp[k], b1 = brp[k + 1];
  if (static_cast<int64_t>(run) != b1 - b0) {  // the chunk counts do not cover the row
    if (lane == 0) set_error(err, kErrBounds);
    return;
  }
  for (int64_t q = b0 + lane; q < b1; q += 32) {
    const int32_t col = bcol[q];
    const int64_t c = static_cast<int64_t>(col) >> shift;
    if (col < 0 || c >= v) {
      set_error(err, kErrBounds);
      continue;
    }
    const int32_t pos = atomicAdd(&cur[c], 1);
    bs_col[b0 + pos] = col;
    if (VALS) bs_val[b0 + pos] = bval[q];
  }
}

void launch_bsplit(const spgemm_csr& B, const int32_t* colcnt, const int32_t* bh, int shift, int64_t v,
                   int32_t* bo, int32_t* bs_col, double* bs_val, uint32_t* err, cudaStream_t s) {
  if (B.rows == 0) return;
  const size_t smem = sizeof(int32_t) * static_cast<size_t>(v) * kBsWarps;
  const unsigned grid = static_cast<unsigned>(ceil_div(B.rows, kBsWarps));
  note_launch();
  if (bs_val) {
    cudaFuncSetAttribute(k_bsplit<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    k_bsplit<true><<<grid, 32 * kBsWarps, smem, s>>>(B.row_ptr, B.col_idx, B.vals, B.rows, colcnt, bh, shift, v, bo,
                                                     bs_col, bs_val, err);
  } else {
    cudaFuncSetAttribute(k_bsplit<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    k_bsplit<false><<<grid, 32 * kBsWarps, smem, s>>>(B.row_ptr, B.col_idx, nullptr, B.rows, colcnt, bh, shift, v,
                                                      bo, bs_col, nullptr, err);
  }
}

// Final chunks of a batch straight from the level-0 counts (row-major counts[p * v + c]),
// enumerated chunk-major (q = c * R + p): the chunks that run together then read the same
// column block of B_split, which stays in L2.  rptr (the exclusive scan of the counts, or null):
// where each chunk's run of C^_reord starts when the numeric phase expands the batch.
__global__ void k_fused_desc(const unsigned long long* __restrict__ counts, const int64_t* __restrict__ rptr,
                             int64_t R, int64_t v, int64_t width, int64_t* __restrict__ fcnt,
                             int32_t* __restrict__ frow, int32_t* __restrict__ fbase, int64_t* __restrict__ fstart) {
  const int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (q >= R * v) return;
  const int64_t c = q / R, p = q - c * R;
  fcnt[q] = static_cast<int64_t>(counts[p * v + c]);
  frow[q] = static_cast<int32_t>(p);
  fbase[q] = static_cast<int32_t>(c * width);
  fstart[q] = rptr ? rptr[p * v + c] : 0;  // nothing stored when the products are generated
}
void launch_fused_desc(const unsigned long long* counts, const int64_t* rptr, int64_t R, int64_t v, int64_t width,
                       int64_t* f_cnt, int32_t* f_row, int32_t* f_base, int64_t* f_start, cudaStream_t s) {
  if (R * v == 0) return;
  note_launch();
  k_fused_desc<<<static_cast<unsigned>(ceil_div(R * v, 256)), 256, 0, s>>>(counts, rptr, R, v, width, f_cnt, f_row,
                                                                          f_base, f_start);
}

// ---- segment table of a batch ---------------------------------------------------------------
// seg[c * E + e] = position in B_split where chunk c of the row of B used by heavy entry e
// starts (c = v: where that row ends), for the E entries of a batch's heavy rows in row order
// (hrp: prefix of the rows' lengths).  Chunk-major, so the chunk tasks of one chunk read their
// entries' ranges coalesced and without a chain of dependent lookups (A column, then B row
// offset, then chunk offset).  Two launches: the A column of every entry (a warp per heavy row,
// one store per entry), then one thread per (entry, group of 32 chunks), consecutive threads on
// consecutive entries, so every store is coalesced and no long row serialises a warp.
__global__ void k_entry_cols(const int64_t* __restrict__ arp, const int32_t* __restrict__ acol,
                             const int32_t* __restrict__ rows, int64_t R, const int64_t* __restrict__ hrp,
                             int32_t* __restrict__ ecol) {
  const int64_t p = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (p >= R) return;
  const int64_t a0 = arp[rows[p]];
  const int64_t e0 = hrp[p];
  const int64_t L = hrp[p + 1] - e0;
  for (int64_t j = lane_id(); j < L; j += 32) ecol[e0 + j] = acol[a0 + j];
}

constexpr int kSegChunks = 32;  // chunks per thread of the segment table

__global__ void k_segtable(const int32_t* __restrict__ ecol, int64_t E, const int64_t* __restrict__ brp,
                           const int32_t* __restrict__ bo, int64_t v, int32_t* __restrict__ seg) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const int32_t k = ecol[e];
  const int32_t b0 = static_cast<int32_t>(brp[k]);
  const int32_t* b = bo + static_cast<int64_t>(k) * (v + 1);
  const int64_t c0 = static_cast<int64_t>(blockIdx.y) * kSegChunks;
  const int64_t c1 = min(v + 1, c0 + kSegChunks);
  for (int64_t c = c0; c < c1; ++c) seg[c * E + e] = b0 + __ldg(&b[c]);
}

void launch_segtable(const spgemm_csr& A, const int32_t* rows, int64_t R, const int64_t* hrp, const spgemm_csr& B,
                     const int32_t* bo, int64_t v, int64_t E, int32_t* ecol, int32_t* seg, cudaStream_t s) {
  if (R == 0 || E == 0) return;
  note_launch();
  k_entry_cols<<<static_cast<unsigned>(ceil_div(R * 32, 256)), 256, 0, s>>>(A.row_ptr, A.col_idx, rows, R, hrp, ecol);
  note_launch();
  const dim3 grid(static_cast<unsigned>(ceil_div(E, 256)), static_cast<unsigned>(ceil_div(v + 1, kSegChunks)));
  k_segtable<<<grid, 256, 0, s>>>(ecol, E, B.row_ptr, bo, v, seg);
}

// The direct split's reservation cursors of a batch whose run starts the symbolic phase kept in
// its descriptors: cursor[row * v + chunk] = f_start of that (row, chunk).
__global__ void k_cursor_from_desc(const int64_t* __restrict__ fstart, const int32_t* __restrict__ frow,
                                   const int32_t* __restrict__ fbase, int64_t n, int64_t v, int shift,
                                   int64_t* __restrict__ cursor) {
  const int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (q < n) cursor[static_cast<int64_t>(frow[q]) * v + (fbase[q] >> shift)] = fstart[q];
}
void launch_cursor_from_desc(const int64_t* f_start, const int32_t* f_row, const int32_t* f_base, int64_t n,
                             int64_t v, int shift, int64_t* cursor, cudaStream_t s) {
  if (n == 0) return;
  note_launch();
  k_cursor_from_desc<<<static_cast<unsigned>(ceil_div(n, 256)), 256, 0, s>>>(f_start, f_row, f_base, n, v, shift,
                                                                             cursor);
}

// ---- product generator -----------------------------------------------------------------------
constexpr int32_t kLongSeg = 16;  // segments of at least this many products are swept lane by entry

// Calls visit(local column, value) once per product of chunk c of a heavy row whose entries are
// [e0, e1) of the batch (A values at aval[abase + e]; value unused without VALS).  Every warp of
// the group walks every window of 32 entries (their loads are cheap and cached); the rounds of
// 32 x U products are dealt out over the warps: the calling warp takes rounds rfirst, rfirst +
// rstep, ... of a count that runs on across segments and windows, so a chunk's products are
// spread evenly over the block even when its row has a single window (the median heavy row of
// R-MAT scale 18 has 28 entries).  Every lane of the warp must call it.  The next window's loads
// are issued before the current window's products, so they are in flight together.
// ROUNDS false: the calling warp takes the windows rfirst, rfirst + rstep, ... and every round of
// them (the symbolic block kernels, whose bitmap updates are cheap next to the loads).
template <bool VALS, bool ROUNDS, typename Visit>
__device__ __forceinline__ void fused_products(const FusedSrc& f, int64_t e0, int64_t e1, int64_t abase, int64_t c,
                                               int32_t base, int rfirst, int rstep, Visit&& visit) {
  const int lane = static_cast<int>(lane_id());
  constexpr int U = 4;  // loads of U x 32 products issued together
  const int32_t* lo_row = f.seg + c * f.E;
  const int32_t* hi_row = lo_row + f.E;
  int32_t nlo = 0, nhi = 0;
  double na = 0.0;
  auto fetch = [&](int64_t ww) {
    const int64_t e = ww + lane;
    nlo = 0;
    nhi = 0;
    if (e < e1) {
      nlo = __ldg(lo_row + e);
      nhi = __ldg(hi_row + e);
      if (VALS) na = __ldg(&f.aval[abase + e]);
    }
  };
  int round = 0;  // the same in every warp of the group
  const int64_t w_first = ROUNDS ? e0 : e0 + static_cast<int64_t>(rfirst) * 32;
  const int64_t w_step = ROUNDS ? 32 : static_cast<int64_t>(rstep) * 32;
  fetch(w_first);
  for (int64_t w = w_first; w < e1; w += w_step) {
    int32_t len = nhi - nlo;
    int32_t qd = nlo;
    const double a = na;
    fetch(w + w_step);
    // long segments (most products of power-law inputs: the long rows of B): consecutive lanes
    // sweep consecutive entries of one segment, no search
    uint32_t longs = __ballot_sync(0xffffffffu, len >= kLongSeg);
    while (longs) {
      const int l = __ffs(longs) - 1;
      longs &= longs - 1;
      const int32_t s0 = __shfl_sync(0xffffffffu, qd, l);
      const int32_t n = __shfl_sync(0xffffffffu, len, l);
      const double al = VALS ? __shfl_sync(0xffffffffu, a, l) : 0.0;
      for (int32_t i0 = 0; i0 < n; i0 += 32 * U, ++round) {
        if (ROUNDS && round % rstep != rfirst) continue;
        int32_t col[U];
        double bv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int32_t i = i0 + 32 * u + lane;
          if (i < n) {
            col[u] = __ldg(&f.bcol[s0 + i]);
            if (VALS) bv[u] = __ldg(&f.bval[s0 + i]);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (i0 + 32 * u + lane < n) visit(col[u] - base, VALS ? al * bv[u] : 0.0);
      }
    }
    if (len >= kLongSeg) len = 0;
    // short segments: flattened over the warp; lane l takes product f0 + l of a round and finds
    // its entry by a binary search over the lanes' inclusive sums
    const int32_t incl = warp_incl_scan(len);
    const int32_t total = __shfl_sync(0xffffffffu, incl, 31);
    qd -= incl - len;  // product fi of this lane's entry sits at B_split position qd + fi
    for (int32_t f0 = 0; f0 < total; f0 += 32 * U, ++round) {
      if (ROUNDS && round % rstep != rfirst) continue;
      int32_t col[U];
      double bv[U], av[U];
      int32_t qq[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int32_t fi = f0 + 32 * u + lane;
        int pos = 0;  // lanes 0 .. pos-1 end at or before fi: the owner of product fi is lane pos
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) {
          if (__shfl_sync(0xffffffffu, incl, pos + d - 1) <= fi) pos += d;
        }
        qq[u] = __shfl_sync(0xffffffffu, qd, pos) + fi;
        if (VALS) av[u] = __shfl_sync(0xffffffffu, a, pos);
        qq[u] = fi < total ? qq[u] : -1;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (qq[u] >= 0) {
          col[u] = __ldg(&f.bcol[qq[u]]);
          if (VALS) bv[u] = __ldg(&f.bval[qq[u]]);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (qq[u] >= 0) visit(col[u] - base, VALS ? av[u] * bv[u] : 0.0);
    }
  }
}

// ---- chunk accumulators on generated products ---------------------------------------------
// mode 0: symbolic (bitmap count), 1: hash numeric; a warp per chunk (8 per block) or a block per
// chunk (its warps share the chunk's windows of A entries).
template <bool WARP, int MODE>
__global__ void __launch_bounds__(WARP ? 32 * kCkWarpsPerBlock : 512) k_fchunk(CkParams p, FusedSrc f) {
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
  const int64_t cnt = p.cs.cnt[q];
  const int64_t grow = p.cs.heavy_rows[p.cs.row[q]];
  if (MODE != 0 && (grow < p.sink.row_begin || grow >= p.sink.row_end)) return;
  const int64_t words = (p.width + 31) / 32;
  const uint32_t width = static_cast<uint32_t>(p.width);
  const int32_t base = p.cs.base[q];
  const int64_t chunk = static_cast<int64_t>(base) >> f.shift;
  uint32_t slots = static_cast<uint32_t>(p.slots);
  if (MODE == 1 && !WARP) {  // table sized for this chunk, as for the expanded chunks
    uint32_t need = 64;
    while (need < 2 * cnt && need < slots) need <<= 1;
    slots = need < slots ? need : slots;
  }
  for (int64_t w = g.lane; w < words; w += g.size) s.bits[w] = 0u;
  if (MODE == 1) {
    for (uint32_t j = g.lane; j < slots; j += g.size) {
      s.keys[j] = kEmptyKey;
      s.vals[j] = 0.0;
    }
  }
  g.sync();
  const int64_t prow = p.cs.row[q];
  const int64_t e0 = f.hrp[prow], e1 = f.hrp[prow + 1];
  const int64_t abase = f.arp[grow] - e0;
  const int rfirst = WARP ? 0 : static_cast<int>(threadIdx.x >> 5);
  const int rstep = WARP ? 1 : static_cast<int>(blockDim.x >> 5);
  uint32_t* err = p.err;
  fused_products<MODE == 1, MODE == 1>(f, e0, e1, abase, chunk, base, rfirst, rstep, [&](int32_t lc, double v) {
    if (static_cast<uint32_t>(lc) >= width) {
      set_error(err, kErrBounds);
      return;
    }
    if (MODE == 0) atomicOr(&s.bits[lc >> 5], 1u << (lc & 31));
    else hash_insert(s, slots, lc, v, err);
  });
  g.sync();
  if (MODE == 0) {
    int64_t n = 0;
    for (int w = g.lane; w < static_cast<int>(words); w += g.size) n += __popc(s.bits[w]);
    int64_t tot;
    ck_scan<WARP>(g, n, s.tmp, &tot);
    if (g.lane == 0) p.cs.nnz[q] = tot;
    return;
  }
  const int64_t out = p.sink.row_ptr[grow] + p.cs.out[q] - p.sink.row_ptr[p.sink.row_begin];
  hash_emit<WARP>(g, s, words, slots, p.cs.nnz[q], base, p.sink.c_col + out, p.sink.c_val + out, p.err);
}

// Dense numeric accumulation on generated products: persistent blocks as in the expanded path
// (k_chunk_dense): warp 0 fetches the next chunk's descriptor while the other warps generate
// and add the current chunk's products; hub columns add into private copies.
struct FusedJob {
  int64_t e0, e1, abase, out, expected;
  int32_t base, state;  // state: 0 none left, 1 work, 2 outside the numeric row window
};

__device__ __forceinline__ void fused_fetch(const CkParams& p, const FusedSrc& f, int* next, FusedJob* j) {
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
  const int64_t prow = p.cs.row[q];
  j->e0 = f.hrp[prow];
  j->e1 = f.hrp[prow + 1];
  j->abase = f.arp[grow] - j->e0;
  j->out = p.sink.row_ptr[grow] + p.cs.out[q] - p.sink.row_ptr[p.sink.row_begin];
  j->expected = p.cs.nnz[q];
  j->base = p.cs.base[q];
  j->state = 1;
}

// One instantiation per block size (256 threads at the default W, 3 blocks per SM; 512 or 1024
// for wider chunks), so that the register budget follows the blocks an SM holds.
template <int THREADS>
__global__ void __launch_bounds__(THREADS, 768 / THREADS > 0 ? 768 / THREADS : 1)
    k_fchunk_dense(CkParams p, FusedSrc f, int* next) {
  extern __shared__ __align__(16) char smem_raw[];
  __shared__ FusedJob jobs[3];
  CkGroup<false> g;
  g.lane = threadIdx.x;
  g.size = blockDim.x;
  const CkSmem s = ck_carve(smem_raw, p.width, 0, 2);
  const int64_t words = (p.width + 31) / 32;
  const uint32_t width = static_cast<uint32_t>(p.width);
  const int warp = threadIdx.x >> 5;
  const int nwork = (blockDim.x >> 5) - 1;
  double* acc = s.vals;
  double* my_hub = s.hub + ((warp > 0 ? warp - 1 : 0) % kHubCopies) * kHubSlots;
  {
    double2* v2 = reinterpret_cast<double2*>(acc);
    for (int64_t j = g.lane; j < p.width / 2; j += g.size) v2[j] = make_double2(0.0, 0.0);
    if ((p.width & 1) && g.lane == 0) acc[p.width - 1] = 0.0;
  }
  for (int j = g.lane; j < kHubCopies * kHubSlots; j += g.size) s.hub[j] = 0.0;
  for (int64_t w = g.lane; w < words; w += g.size) s.bits[w] = 0u;
  if (threadIdx.x == 0) {
    fused_fetch(p, f, next, &jobs[0]);
    if (jobs[0].state != 0) fused_fetch(p, f, next, &jobs[1]);
    else jobs[1].state = 0;
  }
  __syncthreads();
  uint32_t* err = p.err;
  for (int it = 0;; ++it) {
    const FusedJob job = jobs[it % 3];
    if (job.state == 0) break;
    if (warp == 0) {
      if (threadIdx.x == 0) {
        const FusedJob nx = jobs[(it + 1) % 3];
        if (nx.state != 0) fused_fetch(p, f, next, &jobs[(it + 2) % 3]);
        else jobs[(it + 2) % 3].state = 0;
      }
    } else if (job.state == 1) {
      const int64_t chunk = static_cast<int64_t>(job.base) >> f.shift;
      fused_products<true, true>(f, job.e0, job.e1, job.abase, chunk, job.base, warp - 1, nwork,
                           [&](int32_t lc, double v) {
        if (static_cast<uint32_t>(lc) >= width) {
          set_error(err, kErrBounds);
          return;
        }
        atomicOr(&s.bits[lc >> 5], 1u << (lc & 31));
        const int hi = hub_index(static_cast<uint32_t>(lc));
        atomicAdd(hi >= 0 ? &my_hub[hi] : &acc[lc], v);
      });
    }
    __syncthreads();
    if (job.state == 1)
      dense_fold_and_emit<false>(g, s, acc, p.width, job.expected, job.base, p.sink.c_col + job.out,
                                 p.sink.c_val + job.out, p.err);
    __syncthreads();
  }
}

template <bool WARP, int MODE>
static void fck_launch(const CkParams& p, const FusedSrc& f, int tpr, cudaStream_t s) {
  const size_t smem = chunk_smem_bytes(p.width, p.slots, MODE, WARP);
  auto kern = k_fchunk<WARP, MODE>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  const int64_t blocks = WARP ? ceil_div(p.count, kCkWarpsPerBlock) : p.count;
  const int threads = WARP ? 32 * kCkWarpsPerBlock : tpr;
  note_launch();
  kern<<<static_cast<unsigned>(blocks), threads, smem, s>>>(p, f);
}

void launch_fused_chunks(const FusedSrc& f, const ChunkSet& cs, const int32_t* list, int64_t count, int64_t width,
                         int mode, int64_t slots, int tpr, const Sink& sink, uint32_t* err, int* counter,
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
    if (warp) fck_launch<true, 0>(p, f, tpr, s); else fck_launch<false, 0>(p, f, tpr, s);
  } else if (mode == 1) {
    if (warp) fck_launch<true, 1>(p, f, tpr, s); else fck_launch<false, 1>(p, f, tpr, s);
  } else {
    int dev = 0, sms = 0, smem_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaMemsetAsync(counter, 0, sizeof(int), s);
    const size_t smem = chunk_smem_bytes(width, 0, 2, false);
    const int fit = static_cast<int>(smem_sm / (smem + 1024));
    const int threads = fit >= 3 ? 256 : (fit == 2 ? 512 : 1024);
    auto kern = threads == 256 ? k_fchunk_dense<256> : (threads == 512 ? k_fchunk_dense<512> : k_fchunk_dense<1024>);
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    int per_sm = 1;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (per_sm < 1) per_sm = 1;
    const int64_t blocks = std::min<int64_t>(count, static_cast<int64_t>(sms) * per_sm);
    note_launch();
    kern<<<static_cast<unsigned>(blocks), threads, smem, s>>>(p, f, counter);
  }
}

}  // namespace sg
