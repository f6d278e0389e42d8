// Multisplit (gMAGNUS page, section III-C, Algorithm 5) with the tiles of C^ staged in shared
// memory by the bulk-copy (TMA) engine.  Persistent blocks keep two stages: while tile t is
// counted and scattered from one stage, tile t + grid streams into the other, so no thread holds
// a tile in registers and no load sits on the critical path.  Counting, ranking and the scatter
// are those of k_multisplit: the warp-aggregated shared atomics of the count return every
// element's rank inside its bin, one global reservation per bin, then every element is written
// at (its bin's run start + its rank) with the column shifted into the chunk's local range.
//
// Every wait on an mbarrier is bounded: after kMaxSpins failed polls the block records
// kErrTimeout, drains its own copies in flight (again bounded, on the parity of the copy that
// was waited for) and returns.  A test lowers the first wait's limit to reach that path.
#include <algorithm>

#include "internal.h"
#include "ms_tile.cuh"

namespace sg {

namespace {

constexpr int kT = static_cast<int>(kMsTile);  // elements per tile: the partition of k_multisplit
constexpr uint32_t kMaxSpins = 1u << 20;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait; returns false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t spins = kMaxSpins) {
  for (uint32_t i = 0; i < spins; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

struct Stage {
  int32_t* col;
  double* val;
};

// Issue the loads of tile t into stage st: bulk copies of the 16-byte-aligned body; the ragged
// tail (last tile only) is loaded by plain loads after the wait.  Thread 0 only.
template <bool VALS>
__device__ __forceinline__ void issue_tile(const int32_t* in_col, const double* in_val, int64_t total, int64_t t,
                                           Stage st, uint64_t* bar) {
  const int64_t g0 = t * kT;
  const int64_t n = min(static_cast<int64_t>(kT), total - g0);
  const int64_t body = n & ~int64_t(3);  // whole 16-byte groups of columns (and of value pairs)
  const uint32_t cb = static_cast<uint32_t>(body * 4), vb = VALS ? static_cast<uint32_t>(body * 8) : 0u;
  fence_proxy_async();
  mbar_expect_tx(bar, cb + vb);
  if (cb) bulk_g2s(st.col, in_col + g0, cb, bar);
  if (vb) bulk_g2s(st.val, in_val + g0, vb, bar);
}

}  // namespace

template <bool VALS>
__global__ void __launch_bounds__(kMsThreads, 8) k_multisplit_tma(
    const int64_t* __restrict__ rp, const int2* __restrict__ part, int64_t total, int64_t ntiles,
    const int32_t* __restrict__ in_col, const double* __restrict__ in_val, int shift, int64_t v, int64_t gr,
    const int32_t* __restrict__ xmap, unsigned long long* __restrict__ cursor, int32_t* __restrict__ out_col,
    double* __restrict__ out_val, uint32_t* err, uint32_t first_spins) {
  extern __shared__ __align__(128) char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int s_fail;
  // layout (bulk-copy destinations first, all 16-byte aligned): stage 0/1 values | stage 0/1
  // columns | goff | rstart | hist
  const int64_t bins_cap = gr * v;
  char* p = smem_raw;
  double* const val0 = reinterpret_cast<double*>(p);  // stage s: val0 + s * kT
  p += 2 * kT * 8;
  int32_t* const col0 = reinterpret_cast<int32_t*>(p);  // stage s: col0 + s * kT
  p += 2 * kT * 4;
  auto stage = [&](int st) { return Stage{col0 + st * kT, val0 + st * kT}; };
  unsigned long long* goff = reinterpret_cast<unsigned long long*>(p); p += bins_cap * 8;
  int64_t* rstart = reinterpret_cast<int64_t*>(p); p += (gr + 1) * 8;
  unsigned* hist = reinterpret_cast<unsigned*>(p);

  const int64_t wmask = (int64_t(1) << shift) - 1;
  int64_t t = blockIdx.x;
  if (t >= ntiles) return;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    s_fail = 0;
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();
  if (threadIdx.x == 0) {
    issue_tile<VALS>(in_col, in_val, total, t, stage(0), &bars[0]);
    if (t + gridDim.x < ntiles) issue_tile<VALS>(in_col, in_val, total, t + gridDim.x, stage(1), &bars[1]);
  }
  // bit s of `phase`: parity to wait for on stage s; bit s of `pending` (thread 0's view): a copy
  // into stage s was issued and not yet waited for
  uint32_t phase = 0u;
  uint32_t pending = 1u | (t + gridDim.x < ntiles ? 2u : 0u);
  int s = 0;
  bool first = true;
  for (; t < ntiles; t += gridDim.x, s ^= 1) {
    const int64_t g0 = t * kT;
    const int64_t g1 = min(total, g0 + kT);
    const int n = static_cast<int>(g1 - g0);
    const int body = n & ~3;
    const int2 pr = part[t];
    // wait for the stage (bounded; the first wait's limit can be lowered to test the timeout).
    // Thread 0 decides for the block: on a timeout it keeps the stage pending and its parity
    // unflipped, so the drain below waits for that very copy.
    const bool ok = mbar_wait(&bars[s], (phase >> s) & 1u, first ? first_spins : kMaxSpins);
    first = false;
    if (threadIdx.x == 0 && !ok) {
      set_error(err, kErrTimeout);
      s_fail = 1;
    } else {
      pending &= ~(1u << s);
      phase ^= 1u << s;
    }
    const Stage cur = stage(s);
    // ragged tail of the last tile: plain loads
    for (int i = body + static_cast<int>(threadIdx.x); i < n; i += blockDim.x) {
      cur.col[i] = in_col[g0 + i];
      if (VALS) cur.val[i] = in_val[g0 + i];
    }
    __syncthreads();
    if (s_fail) break;
    const int i0 = static_cast<int>(threadIdx.x) * kMsItems;
    const int64_t p0 = g0 + i0;
    int32_t c[kMsItems];
#pragma unroll
    for (int j = 0; j < kMsItems; j += 4) {
      const int4 x = *reinterpret_cast<const int4*>(cur.col + i0 + j);
      c[j] = x.x; c[j + 1] = x.y; c[j + 2] = x.z; c[j + 3] = x.w;
    }
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
      for (int j = 0; j < kMsItems; ++j) rank[j] = ms_rank<true>(hist, bin[j]);
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
#pragma unroll
      for (int j = 0; j < kMsItems; ++j) {
        const int b = bin[j];
        if (b >= 0) {
          const int64_t dst = static_cast<int64_t>(goff[b]) + rank[j];
          __stcs(&out_col[dst], static_cast<int32_t>(c[j] & wmask));
          if (VALS) __stcs(&out_val[dst], cur.val[i0 + j]);
        }
      }
    }
    __syncthreads();  // every read of stage s is done: it may be refilled
    if (threadIdx.x == 0 && t + 2 * static_cast<int64_t>(gridDim.x) < ntiles) {
      issue_tile<VALS>(in_col, in_val, total, t + 2 * gridDim.x, cur, &bars[s]);
      pending |= 1u << s;
    }
  }
  // drain: after a timeout, wait (bounded) for this block's copies still in flight before exiting
  if (threadIdx.x == 0) {
    for (int k = 0; k < 2; ++k)
      if ((pending >> k) & 1u) (void)mbar_wait(&bars[k], (phase >> k) & 1u);
  }
}

size_t multisplit_tma_smem(int64_t group_rows, int64_t nchunks) {
  const int64_t bins = group_rows * nchunks;
  return static_cast<size_t>(2 * kT * 8 + 2 * kT * 4 + bins * 8 + (group_rows + 1) * 8 + bins * 4);
}

bool launch_multisplit_tma(const int64_t* row_ptr, const int2* part, int64_t total, const int32_t* in_col,
                           const double* in_val, int shift, int64_t nchunks, int64_t group_rows, const int32_t* xmap,
                           unsigned long long* cursor, int32_t* out_col, double* out_val, bool with_vals, int sms,
                           uint32_t* err, cudaStream_t s, uint32_t first_spins) {
  if (total == 0) return true;
  const size_t smem = multisplit_tma_smem(group_rows, nchunks);
  if (smem > 227 * 1024) return false;  // too many bins for this variant
  // bulk copies need 16-byte aligned sources
  if ((reinterpret_cast<uintptr_t>(in_col) & 15) || (with_vals && (reinterpret_cast<uintptr_t>(in_val) & 15)))
    return false;
  const int64_t ntiles = ceil_div(total, static_cast<int64_t>(kT));
  auto kern = with_vals ? k_multisplit_tma<true> : k_multisplit_tma<false>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kMsThreads, smem);
  if (per_sm < 1) per_sm = 1;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(ntiles, static_cast<int64_t>(sms) * per_sm));
  note_launch();
  kern<<<grid, kMsThreads, smem, s>>>(row_ptr, part, total, ntiles, in_col, with_vals ? in_val : nullptr, shift,
                                      nchunks, group_rows, xmap, cursor, out_col, with_vals ? out_val : nullptr, err,
                                      first_spins ? first_spins : kMaxSpins);
  return true;
}

}  // namespace sg
