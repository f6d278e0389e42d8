// Multisplit (gMAGNUS page, section III-C, Algorithm 5) with the tiles of C^ staged in shared
// memory by the bulk-copy (TMA) engine.  Persistent blocks, one per SM; tile t is processed while
// tile t + gridDim.x streams into the second stage, so global loads never sit on the critical path.
// Per tile: local histogram over (row, chunk) bins with warp-aggregated updates, exclusive scan,
// one global reservation per non-empty bin, permute in shared memory, and a coalesced write of
// every local chunk run with the column shifted into the chunk's range.
//
// Every wait on an mbarrier is bounded: after kMaxSpins failed polls the block records
// kErrTimeout, drains its own copies in flight (again bounded) and returns.
#include <algorithm>

#include "internal.h"

namespace sg {

namespace {

constexpr int kT = static_cast<int>(kMsTile);   // 4096 elements per tile
constexpr int kThreads = 1024;
constexpr int kItems = kT / kThreads;            // 4
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
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kMaxSpins; ++i)
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
__global__ void __launch_bounds__(kThreads, 1) k_multisplit_tma(
    const int64_t* __restrict__ rp, const int2* __restrict__ part, int64_t total, int64_t ntiles,
    const int32_t* __restrict__ in_col, const double* __restrict__ in_val, int shift, int64_t v, int64_t gr,
    const int32_t* __restrict__ xmap, unsigned long long* __restrict__ cursor, int32_t* __restrict__ out_col,
    double* __restrict__ out_val, uint32_t* err) {
  extern __shared__ __align__(128) char smem_raw[];
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ unsigned scan_tmp[33];
  __shared__ int s_fail;
  // layout (bulk-copy destinations first, all 16-byte aligned): stage 0/1 vals | stage 0/1 cols |
  // permuted vals | permuted cols | goff | rstart | hist | loff
  const int64_t bins_cap = gr * v;
  char* p = smem_raw;
  Stage stg[2];
  stg[0].val = reinterpret_cast<double*>(p); p += kT * 8;
  stg[1].val = reinterpret_cast<double*>(p); p += kT * 8;
  stg[0].col = reinterpret_cast<int32_t*>(p); p += kT * 4;
  stg[1].col = reinterpret_cast<int32_t*>(p); p += kT * 4;
  double* val_buf = reinterpret_cast<double*>(p); p += kT * 8;
  int32_t* col_buf = reinterpret_cast<int32_t*>(p); p += kT * 4;
  unsigned long long* goff = reinterpret_cast<unsigned long long*>(p); p += bins_cap * 8;
  int64_t* rstart = reinterpret_cast<int64_t*>(p); p += (gr + 1) * 8;
  unsigned* hist = reinterpret_cast<unsigned*>(p); p += bins_cap * 4;
  unsigned* loff = reinterpret_cast<unsigned*>(p);

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
    issue_tile<VALS>(in_col, in_val, total, t, stg[0], &bars[0]);
    if (t + gridDim.x < ntiles) issue_tile<VALS>(in_col, in_val, total, t + gridDim.x, stg[1], &bars[1]);
  }
  uint32_t phase[2] = {0u, 0u};
  int pending[2] = {1, t + gridDim.x < ntiles ? 1 : 0};  // thread 0's view: copies issued, not yet waited
  int s = 0;
  for (; t < ntiles; t += gridDim.x, s ^= 1) {
    const int64_t g0 = t * kT;
    const int64_t g1 = min(total, g0 + kT);
    const int n = static_cast<int>(g1 - g0);
    const int body = n & ~3;
    // wait for the stage (bounded)
    if (!mbar_wait(&bars[s], phase[s])) {
      if (threadIdx.x == 0) {
        set_error(err, kErrTimeout);
        s_fail = 1;
      }
    } else {
      pending[s] = 0;
    }
    phase[s] ^= 1u;
    // ragged tail of the last tile: plain loads
    for (int i = body + static_cast<int>(threadIdx.x); i < n; i += blockDim.x) {
      stg[s].col[i] = in_col[g0 + i];
      if (VALS) stg[s].val[i] = in_val[g0 + i];
    }
    __syncthreads();
    if (s_fail) break;
    const int2 pr = part[t];
    const int32_t* scol = stg[s].col;
    const double* sval = stg[s].val;
    for (int64_t w0 = pr.x; w0 <= pr.y; w0 += gr) {
      const int nr = static_cast<int>(min(gr, static_cast<int64_t>(pr.y) - w0 + 1));
      const int nbins = static_cast<int>(nr * v);
      for (int i = threadIdx.x; i <= nr; i += blockDim.x) rstart[i] = rp[w0 + i] - g0;  // tile-relative
      for (int i = threadIdx.x; i < nbins; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      const int64_t e0 = max(int64_t(0), rstart[0]);
      const int64_t e1 = min(static_cast<int64_t>(n), rstart[nr]);
      int bin[kItems];
#pragma unroll
      for (int j = 0; j < kItems; ++j) {
        const int i = static_cast<int>(threadIdx.x) + j * kThreads;
        int b = -1;
        if (i >= e0 && i < e1) {
          int r = 0;
          while (r + 1 < nr && i >= rstart[r + 1]) ++r;
          const int64_t ch = static_cast<int64_t>(scol[i]) >> shift;
          if (ch < v) b = static_cast<int>(r * v + ch);
          else set_error(err, kErrBounds);
        }
        bin[j] = b;
        const uint32_t peers = __match_any_sync(0xffffffffu, b);
        if (b >= 0 && (peers & lanemask_lt()) == 0) atomicAdd(&hist[b], __popc(peers));
      }
      __syncthreads();
      {
        const int per = (nbins + kThreads - 1) / kThreads;
        const int b0 = threadIdx.x * per;
        unsigned local = 0;
        for (int b = b0; b < min(nbins, b0 + per); ++b) local += hist[b];
        unsigned tot;
        const unsigned incl = block_incl_scan(local, scan_tmp, &tot);
        unsigned run = incl - local;
        for (int b = b0; b < min(nbins, b0 + per); ++b) {
          const unsigned h = hist[b];
          loff[b] = run;
          if (h) {
            const int64_t gchunk = (w0 + b / v) * v + (b % v);
            const int64_t q = xmap ? xmap[gchunk] : gchunk;
            goff[b] = atomicAdd(&cursor[q], static_cast<unsigned long long>(h));
          }
          hist[b] = run;
          run += h;
        }
        if (threadIdx.x == 0) loff[nbins] = tot;
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kItems; ++j) {
        const int i = static_cast<int>(threadIdx.x) + j * kThreads;
        const int b = bin[j];
        const uint32_t peers = __match_any_sync(0xffffffffu, b);
        const int leader = __ffs(peers) - 1;
        unsigned base = 0;
        if (b >= 0 && static_cast<int>(lane_id()) == leader) base = atomicAdd(&hist[b], __popc(peers));
        base = __shfl_sync(0xffffffffu, base, leader);
        if (b >= 0) {
          const unsigned pos = base + __popc(peers & lanemask_lt());
          col_buf[pos] = scol[i];
          if (VALS) val_buf[pos] = sval[i];
        }
      }
      __syncthreads();
      const bool last_window = w0 + gr > pr.y;
      if (last_window && threadIdx.x == 0 && t + 2 * static_cast<int64_t>(gridDim.x) < ntiles) {
        issue_tile<VALS>(in_col, in_val, total, t + 2 * gridDim.x, stg[s], &bars[s]);  // stage s is free
        pending[s] = 1;
      }
      const int cnt = static_cast<int>(loff[nbins]);
      for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
        const int32_t cc = col_buf[i];
        int r = 0;
        {
          int lo = 0, hi = nr - 1;
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (static_cast<int>(loff[mid * v]) <= i) lo = mid; else hi = mid - 1;
          }
          r = lo;
        }
        const int b = static_cast<int>(r * v + (static_cast<int64_t>(cc) >> shift));
        const int64_t dst = static_cast<int64_t>(goff[b]) + (i - static_cast<int>(loff[b]));
        __stcs(&out_col[dst], static_cast<int32_t>(cc & wmask));
        if (VALS) __stcs(&out_val[dst], val_buf[i]);
      }
      __syncthreads();
    }
  }
  // drain: after a timeout, wait (bounded) for this block's copies still in flight before exiting
  if (threadIdx.x == 0) {
    for (int k = 0; k < 2; ++k)
      if (pending[k]) (void)mbar_wait(&bars[k], phase[k]);
  }
}

size_t multisplit_tma_smem(int64_t group_rows, int64_t nchunks) {
  const int64_t bins = group_rows * nchunks;
  return static_cast<size_t>(3 * kT * 8 + bins * 8 + (group_rows + 1) * 8 + 3 * kT * 4 + bins * 4 + (bins + 1) * 4);
}

bool launch_multisplit_tma(const int64_t* row_ptr, const int2* part, int64_t total, const int32_t* in_col,
                           const double* in_val, int shift, int64_t nchunks, int64_t group_rows, const int32_t* xmap,
                           unsigned long long* cursor, int32_t* out_col, double* out_val, bool with_vals, int sms,
                           uint32_t* err, cudaStream_t s) {
  if (total == 0) return true;
  const size_t smem = multisplit_tma_smem(group_rows, nchunks);
  if (smem > 227 * 1024) return false;  // too many bins for this variant
  // bulk copies need 16-byte aligned sources
  if ((reinterpret_cast<uintptr_t>(in_col) & 15) || (with_vals && (reinterpret_cast<uintptr_t>(in_val) & 15)))
    return false;
  const int64_t ntiles = ceil_div(total, static_cast<int64_t>(kT));
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(ntiles, sms));
  note_launch();
  if (with_vals) {
    cudaFuncSetAttribute(k_multisplit_tma<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    k_multisplit_tma<true><<<grid, kThreads, smem, s>>>(row_ptr, part, total, ntiles, in_col, in_val, shift, nchunks,
                                                        group_rows, xmap, cursor, out_col, out_val, err);
  } else {
    cudaFuncSetAttribute(k_multisplit_tma<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    k_multisplit_tma<false><<<grid, kThreads, smem, s>>>(row_ptr, part, total, ntiles, in_col, nullptr, shift,
                                                         nchunks, group_rows, xmap, cursor, out_col, nullptr, err);
  }
  return true;
}

}  // namespace sg
