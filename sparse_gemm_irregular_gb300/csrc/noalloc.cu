// spgemm_symbolic_noalloc: C.row_ptr of a light product without any device allocation.
//
// Who needs this: callers that cannot call cudaMalloc (or any allocator) at the moment they
// need the row sizes of C -- for example code running inside a custom allocator or a memory
// manager that is itself servicing an allocation, real-time or embedded loops that forbid
// allocation after start-up, and hosts that hand the library a fixed memory budget.  The
// regular spgemm_create / spgemm_symbolic path allocates its workspace (bins, scan scratch,
// intermediate buffers) with cudaMallocAsync; this entry point instead uses one file-scope
// __device__ array.  Under CUDA's lazy module loading the array and the four kernels below
// come into device memory with the first call on each device (that call's symbol lookup and
// launches load the module), so the first call may itself take device memory: make one
// warm-up call per device at start-up (m = 0 suffices), before any stream capture and before
// entering code that must not allocate.  Later calls allocate nothing.
//
// Scope and limits:
//   * every row of A*B may have at most kNaMaxRowIP intermediate products (the warp hash
//     below holds twice that many columns); a row above it makes the call fail;
//   * A has at most kNaMaxRows rows (the scan keeps one partial sum per 4096 rows in the
//     static array, and the partial sums are scanned by one block).
// Device memory held: sizeof(g_na_scratch) = 33,280 bytes on every device that loads the
// library, until the process exits.
#include <mutex>

#include "internal.h"

namespace {

constexpr int64_t kNaTile = 4096;                 // rows per scan tile (512 threads x 8)
constexpr int64_t kNaMaxTiles = 4096;             // partial sums one block scans
constexpr int64_t kNaMaxRows = kNaTile * kNaMaxTiles - 1;
constexpr int64_t kNaMaxRowIP = 2048;
constexpr int kNaSlots = 2 * kNaMaxRowIP;         // hash slots per warp (load factor <= 1/2)
constexpr int kNaWarps = 4;                       // rows per block
constexpr int kNaScanThreads = 512;
constexpr int kNaItems = static_cast<int>(kNaTile) / kNaScanThreads;

// [0, kNaMaxTiles): partial sums of the scan tiles; [kNaMaxTiles]: total;
// [kNaMaxTiles + 1]: error flags.  Shared by every call on the device.
constexpr int64_t kNaScratchElems = kNaMaxTiles + 64;
static __device__ __align__(256) int64_t g_na_scratch[kNaScratchElems];

constexpr uint32_t kNaErrRowTooLong = 1u;
constexpr uint32_t kNaErrHashFull = 2u;
constexpr uint32_t kNaErrBounds = 4u;   // a row pointer or column index outside its range

__device__ __forceinline__ void na_flag(int64_t* scratch, uint32_t bit) {
  atomicOr(reinterpret_cast<unsigned long long*>(&scratch[kNaMaxTiles + 1]), bit);
}

// One warp per row: distinct columns of row i of A*B, counted in a shared-memory hash.
// Malformed input (a row pointer outside [0, nnz] or decreasing, a column outside its range)
// is skipped and flagged, never read past.
__global__ void __launch_bounds__(32 * kNaWarps) k_na_row_nnz(
    const int64_t* __restrict__ arp, const int32_t* __restrict__ acol, int64_t a_nnz, const int64_t* __restrict__ brp,
    const int32_t* __restrict__ bcol, int64_t b_nnz, int64_t k_dim, int64_t n_dim, int64_t m,
    int64_t* __restrict__ out, int64_t* scratch) {
  extern __shared__ int32_t na_keys[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kNaWarps + warp;
  if (blockIdx.x == 0 && threadIdx.x == 0) out[m] = 0;
  if (row >= m) return;
  int32_t* keys = na_keys + warp * kNaSlots;
  const int64_t a0 = arp[row], a1 = arp[row + 1];
  if (a0 < 0 || a1 < a0 || a1 > a_nnz) {
    if (lane == 0) {
      na_flag(scratch, kNaErrBounds);
      out[row] = 0;
    }
    return;
  }
  // B row k as a checked range: empty (and flagged) when k or its row pointers are out of range
  auto brow = [&](int32_t k, int64_t& b0, int64_t& b1) {
    b0 = b1 = 0;
    if (k < 0 || k >= k_dim) {
      na_flag(scratch, kNaErrBounds);
      return;
    }
    const int64_t s = brp[k], e = brp[k + 1];
    if (s < 0 || e < s || e > b_nnz) {
      na_flag(scratch, kNaErrBounds);
      return;
    }
    b0 = s;
    b1 = e;
  };
  int64_t ip = 0;
  for (int64_t e = a0 + lane; e < a1; e += 32) {
    int64_t b0, b1;
    brow(acol[e], b0, b1);
    ip += b1 - b0;
  }
  ip = sg::warp_sum(ip);
  if (ip > kNaMaxRowIP) {
    if (lane == 0) {
      na_flag(scratch, kNaErrRowTooLong);
      out[row] = 0;
    }
    return;
  }
  for (int j = lane; j < kNaSlots; j += 32) keys[j] = sg::kEmptyKey;
  __syncwarp();
  int64_t fresh = 0;
  for (int64_t e = a0; e < a1; ++e) {
    int64_t b0, b1;
    brow(acol[e], b0, b1);
    for (int64_t q = b0 + lane; q < b1; q += 32) {
      const int32_t c = bcol[q];
      if (c < 0 || c >= n_dim) {
        na_flag(scratch, kNaErrBounds);
        continue;
      }
      uint32_t slot = sg::hash_slot(c, kNaSlots);
      bool done = false;
      for (int probe = 0; probe < kNaSlots && !done; ++probe) {
        const int32_t cur = *reinterpret_cast<volatile int32_t*>(&keys[slot]);
        if (cur == c) {
          done = true;
        } else if (cur == sg::kEmptyKey) {
          const int32_t old = atomicCAS(&keys[slot], sg::kEmptyKey, c);
          if (old == sg::kEmptyKey) {
            ++fresh;
            done = true;
          } else if (old == c) {
            done = true;
          }
        }
        if (!done) slot = (slot + 1 == kNaSlots) ? 0 : slot + 1;
      }
      if (!done) na_flag(scratch, kNaErrHashFull);
    }
  }
  fresh = sg::warp_sum(fresh);
  if (lane == 0) out[row] = fresh;
}

__global__ void __launch_bounds__(kNaScanThreads) k_na_tile_sums(const int64_t* __restrict__ v, int64_t n,
                                                                 int64_t* scratch) {
  __shared__ int64_t tmp[32];
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kNaTile;
  int64_t s = 0;
  for (int j = 0; j < kNaItems; ++j) {
    const int64_t i = base + j * kNaScanThreads + threadIdx.x;
    if (i < n) s += v[i];
  }
  s = sg::warp_sum(s);
  if ((threadIdx.x & 31) == 0) tmp[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    int64_t w = threadIdx.x < kNaScanThreads / 32 ? tmp[threadIdx.x] : 0;
    w = sg::warp_sum(w);
    if (threadIdx.x == 0) scratch[blockIdx.x] = w;
  }
}

// One block: exclusive scan of the nb partial sums in place; the total goes to scratch[kNaMaxTiles].
__global__ void __launch_bounds__(kNaScanThreads) k_na_scan_sums(int64_t nb, int64_t* scratch) {
  __shared__ int64_t tmp[33];
  const int64_t base = threadIdx.x * kNaItems;
  int64_t v[kNaItems];
  int64_t local = 0;
  for (int j = 0; j < kNaItems; ++j) {
    v[j] = base + j < nb ? scratch[base + j] : 0;
    local += v[j];
  }
  int64_t tot;
  const int64_t incl = sg::block_incl_scan(local, tmp, &tot);
  int64_t run = incl - local;
  for (int j = 0; j < kNaItems; ++j) {
    if (base + j < nb) scratch[base + j] = run;
    run += v[j];
  }
  if (threadIdx.x == 0) scratch[kNaMaxTiles] = tot;
}

__global__ void __launch_bounds__(kNaScanThreads) k_na_tile_scan(int64_t* v, int64_t n, const int64_t* scratch) {
  __shared__ int64_t tmp[33];
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kNaTile + threadIdx.x * kNaItems;
  int64_t x[kNaItems];
  int64_t local = 0;
  for (int j = 0; j < kNaItems; ++j) {
    x[j] = base + j < n ? v[base + j] : 0;
    local += x[j];
  }
  int64_t tot;
  const int64_t incl = sg::block_incl_scan(local, tmp, &tot);
  int64_t run = incl - local + scratch[blockIdx.x];
  for (int j = 0; j < kNaItems; ++j) {
    if (base + j < n) v[base + j] = run;
    run += x[j];
  }
}

// Device address of g_na_scratch, looked up once per device (with that device current).
std::mutex g_na_mutex;
int64_t* g_na_ptr[64] = {nullptr};

int na_scratch(int64_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return sg::check_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) {
    sg::set_last_error("device ordinal beyond 63");
    return SPGEMM_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lock(g_na_mutex);
  if (!g_na_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_na_scratch);
    if (e != cudaSuccess) return sg::check_cuda(e, "cudaGetSymbolAddress(g_na_scratch)");
    g_na_ptr[dev] = static_cast<int64_t*>(p);
  }
  *out = g_na_ptr[dev];
  return SPGEMM_OK;
}

}  // namespace

extern "C" int spgemm_symbolic_noalloc(int64_t m, int64_t k, int64_t n, const spgemm_csr* A,
                                       const spgemm_csr* B, int64_t* c_row_ptr, int64_t* c_nnz,
                                       void* stream) {
  sg::set_last_error("");
  if (!A || !B || !c_row_ptr || !c_nnz || m < 0 || k < 0 || n < 0) {
    sg::set_last_error("null pointer or negative size");
    return SPGEMM_ERR_INVALID_ARG;
  }
  if (A->rows != m || A->cols != k || B->rows != k || B->cols != n || !A->row_ptr || !B->row_ptr ||
      (A->nnz > 0 && !A->col_idx) || (B->nnz > 0 && !B->col_idx)) {
    sg::set_last_error("shapes or CSR descriptors do not match");
    return SPGEMM_ERR_INVALID_ARG;
  }
  if (m > kNaMaxRows) {
    sg::set_last_error("spgemm_symbolic_noalloc: A has more than 16,777,215 rows");
    return SPGEMM_ERR_INVALID_ARG;
  }
  if (n > 0x7fffffffLL || k > 0x7fffffffLL) {
    sg::set_last_error("dimensions beyond int32 indices");
    return SPGEMM_ERR_OVERFLOW;
  }
  int64_t* scratch = nullptr;
  int rc = na_scratch(&scratch);
  if (rc != SPGEMM_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the error flags must start at zero; the partial sums are fully rewritten
  rc = sg::check_cuda(cudaMemsetAsync(scratch + kNaMaxTiles + 1, 0, sizeof(int64_t), st), "clear flags");
  if (rc != SPGEMM_OK) return rc;
  const size_t smem = static_cast<size_t>(kNaWarps) * kNaSlots * sizeof(int32_t);
  rc = sg::check_cuda(cudaFuncSetAttribute(k_na_row_nnz, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem)), "smem attribute");
  if (rc != SPGEMM_OK) return rc;
  const unsigned blocks = static_cast<unsigned>(sg::ceil_div(m > 0 ? m : 1, kNaWarps));
  k_na_row_nnz<<<blocks, 32 * kNaWarps, smem, st>>>(A->row_ptr, A->col_idx, A->nnz, B->row_ptr, B->col_idx,
                                                      B->nnz, k, n, m, c_row_ptr, scratch);
  const int64_t len = m + 1;
  const int64_t nb = sg::ceil_div(len, kNaTile);
  k_na_tile_sums<<<static_cast<unsigned>(nb), kNaScanThreads, 0, st>>>(c_row_ptr, len, scratch);
  k_na_scan_sums<<<1, kNaScanThreads, 0, st>>>(nb, scratch);
  k_na_tile_scan<<<static_cast<unsigned>(nb), kNaScanThreads, 0, st>>>(c_row_ptr, len, scratch);
  // launch errors of these four kernels, before anything else is enqueued
  rc = sg::check_cuda(cudaGetLastError(), "spgemm_symbolic_noalloc launch");
  if (rc != SPGEMM_OK) return rc;
  int64_t flags = 0, nnz = 0;
  rc = sg::check_cuda(cudaMemcpyAsync(&flags, scratch + kNaMaxTiles + 1, sizeof(int64_t),
                                      cudaMemcpyDeviceToHost, st), "copy flags");
  if (rc != SPGEMM_OK) return rc;
  rc = sg::check_cuda(cudaMemcpyAsync(&nnz, c_row_ptr + m, sizeof(int64_t), cudaMemcpyDeviceToHost, st),
                      "copy nnz");
  if (rc != SPGEMM_OK) return rc;
  rc = sg::check_cuda(cudaStreamSynchronize(st), "spgemm_symbolic_noalloc");
  if (rc != SPGEMM_OK) return rc;
  if (flags & kNaErrBounds) {
    sg::set_last_error("spgemm_symbolic_noalloc: a row pointer or column index of A or B is out of range");
    return SPGEMM_ERR_INVALID_ARG;
  }
  if (flags & kNaErrRowTooLong) {
    sg::set_last_error("spgemm_symbolic_noalloc: a row of A*B has more than 2048 intermediate products");
    return SPGEMM_ERR_INVALID_ARG;
  }
  if (flags & kNaErrHashFull) {
    sg::set_last_error("spgemm_symbolic_noalloc: hash table full");
    return SPGEMM_ERR_DEVICE;
  }
  *c_nnz = nnz;
  return SPGEMM_OK;
}
