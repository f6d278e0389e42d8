// C ABI and orchestration of the gMAGNUS pipeline (gMAGNUS page, Algorithm 3).
//
//   create    : planner, IP per row + bins (light ladder / heavy), one synchronisation.
//   symbolic  : light rows (hash / shortened dense symbolic), heavy batches (CSC -> level-0
//               histogram from per-B-row chunk counts -> outer product -> levels of histogram +
//               partition + multisplit -> chunk symbolic), scan of C.row_ptr, one
//               synchronisation for nnz(C).
//   numeric   : light rows (accumulate + ordered write), heavy batches (chunk accumulate +
//               ordered write at the final positions).  The expansion is kept from symbolic
//               to numeric when the whole heavy part fits one batch ("resident"), otherwise
//               it is recomputed batch by batch (the device cannot hold C^ of every heavy row
//               of the largest products).  numeric_rows computes a row window;
//               numeric_host streams row windows into host memory.  A repeated numeric call
//               replays a CUDA graph captured on its second occurrence.
//   light-row workflows (Ocean page, Table 1): the exact symbolic pass above, or the light rows
//               accumulated during symbolic into slots sized by their IP bound or by HyperLogLog
//               estimates (with a fallback pass for rows that overflow), copied out in numeric.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <memory>
#include <mutex>
#include <string>

#include "internal.h"

static thread_local std::string g_last_error;
static std::atomic<long long> g_launches{0};

namespace sg {

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
long long launch_count() { return g_launches.load(std::memory_order_relaxed); }

void set_last_error(const std::string& s) { g_last_error = s; }

int check_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return SPGEMM_OK;
  set_last_error(std::string(what) + ": " + cudaGetErrorString(e));
  return SPGEMM_ERR_CUDA;
}

// Workspace comes from one stream-ordered memory pool per device that keeps freed memory for
// reuse (release threshold = unlimited): products of the same size then allocate without
// mapping new physical memory.  spgemm_release_memory() hands the cached memory back.
static std::mutex g_pool_mu;
static cudaMemPool_t g_pool[64] = {};

cudaMemPool_t device_pool(int dev) {
  std::lock_guard<std::mutex> lock(g_pool_mu);
  if (dev < 0 || dev >= 64) return nullptr;
  if (!g_pool[dev]) {
    cudaMemPoolProps props;
    memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    uint64_t thr = ~0ull;
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &thr);
    g_pool[dev] = pool;
  }
  return g_pool[dev];
}

void* ws_alloc(spgemm_ctx* h, size_t bytes) {
  void* p = nullptr;
  if (h->capturing) return nullptr;  // a captured phase must not allocate: the capture is dropped
  if (bytes == 0) bytes = 16;
  if (h->opt.workspace_limit > 0 && h->ws_bytes + bytes > static_cast<size_t>(h->opt.workspace_limit))
    return nullptr;  // the caller's budget
  if (cudaMallocFromPoolAsync(&p, bytes, h->pool, h->st) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  h->allocs.push_back(p);
  h->alloc_bytes.push_back(bytes);
  h->ws_bytes += bytes;
  return p;
}

void ws_free(spgemm_ctx* h, void* p) {
  if (!p) return;
  auto it = std::find(h->allocs.begin(), h->allocs.end(), p);
  if (it != h->allocs.end()) {
    const size_t i = static_cast<size_t>(it - h->allocs.begin());
    h->ws_bytes -= h->alloc_bytes[i];
    h->alloc_bytes.erase(h->alloc_bytes.begin() + static_cast<std::ptrdiff_t>(i));
    h->allocs.erase(it);
  }
  cudaFreeAsync(p, h->st);
}

// Streams and events outlive their handles: a process-wide free list per device, so that small
// products do not pay for creating and destroying them.  A pooled stream is idle when returned
// (its handle synchronised it).
static std::mutex g_sp_mu;
static std::vector<cudaStream_t> g_sp_streams[64];
static std::vector<cudaEvent_t> g_sp_events[64];

cudaStream_t pooled_stream(int dev) {
  {
    std::lock_guard<std::mutex> lock(g_sp_mu);
    if (dev >= 0 && dev < 64 && !g_sp_streams[dev].empty()) {
      cudaStream_t s = g_sp_streams[dev].back();
      g_sp_streams[dev].pop_back();
      return s;
    }
  }
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return s;
}

cudaEvent_t pooled_event(int dev) {
  {
    std::lock_guard<std::mutex> lock(g_sp_mu);
    if (dev >= 0 && dev < 64 && !g_sp_events[dev].empty()) {
      cudaEvent_t e = g_sp_events[dev].back();
      g_sp_events[dev].pop_back();
      return e;
    }
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return e;
}

void return_stream(int dev, cudaStream_t s) {
  if (!s) return;
  std::lock_guard<std::mutex> lock(g_sp_mu);
  if (dev >= 0 && dev < 64) g_sp_streams[dev].push_back(s);
  else cudaStreamDestroy(s);
}

void return_event(int dev, cudaEvent_t e) {
  if (!e) return;
  std::lock_guard<std::mutex> lock(g_sp_mu);
  if (dev >= 0 && dev < 64) g_sp_events[dev].push_back(e);
  else cudaEventDestroy(e);
}

// Page-locked status block of the calling thread: the device error word, nnz(C) and the numeric
// bin starts land here by asynchronous copies, so one synchronisation reads them all.  The calls
// of one thread are sequential, so one block per thread suffices.  Null if it cannot be had.
struct HostStatus {
  uint32_t err;
  uint32_t pad;
  int64_t nnz;
  int64_t starts[kMaxLadder + 1];
};

HostStatus* host_status() {
  thread_local HostStatus* hs = nullptr;
  thread_local bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    if (cudaMallocHost(&p, sizeof(HostStatus)) == cudaSuccess) hs = static_cast<HostStatus*>(p);
    else cudaGetLastError();
  }
  return hs;
}

Ladder make_ladder(int64_t tau) {
  Ladder L;
  int64_t u = 32;
  while (u < tau && u <= 4096 && L.n < kMaxLadder - 1) {
    L.upper[L.n++] = u;
    u *= 2;
  }
  L.upper[L.n++] = tau;
  for (int i = 0; i < L.n; ++i) {
    const int64_t up = L.upper[i];
    L.slots[i] = 2 * up;
    // threads per row: a warp up to 256 products, then blocks about a quarter the size of the
    // bin's products (smaller blocks keep more rows in flight per SM; halving the earlier
    // 256/512/1024 ladder saved 2.4 ms of light-row time on R-MAT s18)
    L.tpr[i] = up <= 256 ? 32 : (up <= 512 ? 128 : (up <= 1024 ? 256 : (up <= 4096 ? 512 : 1024)));
  }
  return L;
}

}  // namespace sg

using namespace sg;

#define SG_TRY(expr)                 \
  do {                               \
    int _rc = (expr);                \
    if (_rc != SPGEMM_OK) return _rc; \
  } while (0)

#define SG_ALLOC(ptr, type, count)                                                     \
  do {                                                                                 \
    ptr = static_cast<type*>(ws_alloc(h, sizeof(type) * static_cast<size_t>(count))); \
    if (!ptr) {                                                                        \
      set_last_error("device workspace allocation failed (" #ptr ")");                \
      return SPGEMM_ERR_OUT_OF_MEMORY;                                                 \
    }                                                                                  \
  } while (0)

namespace {

// Last-level chunk bins: threads per chunk and hash slots (bin 3 is the dense accumulator).
constexpr int kChunkTpr[4] = {32, 256, 512, 1024};
constexpr int kChunkSymTpr[4] = {32, 128, 128, 128};  // symbolic: bitmap only, many small blocks per SM
// symbolic on generated products: chunks of up to 1024 products on one warp as well (R-MAT scale
// 21, same box: 559 -> 525 ms; 64-thread blocks for the larger bins measured slower, 637 ms)
constexpr int kFusedSymTpr[4] = {32, 32, 128, 128};
constexpr int64_t kChunkSlots[4] = {512, 2048, 2 * kChunkDenseMin, 0};

// Scan scratch that grows on demand.
int64_t* scan_scratch(spgemm_ctx* h, int64_t n) {
  const int64_t need = scan_scratch_elems(n);
  if (need > h->scan_cap) {
    ws_free(h, h->d_scan);
    h->d_scan = static_cast<int64_t*>(ws_alloc(h, sizeof(int64_t) * need));
    h->scan_cap = h->d_scan ? need : 0;
  }
  return h->d_scan;
}

int scan(spgemm_ctx* h, const int64_t* in, int64_t* out, int64_t n) {
  int64_t* sc = scan_scratch(h, n);
  if (!sc) {
    set_last_error("scan scratch allocation failed");
    return SPGEMM_ERR_OUT_OF_MEMORY;
  }
  scan_excl_i64(in, out, n, sc, h->st);
  return SPGEMM_OK;
}

int sync_and_check(spgemm_ctx* h, const char* where) {
  uint32_t err = 0;
  HostStatus* hs = host_status();
  if (hs) {  // the error word rides on the same synchronisation
    SG_TRY(check_cuda(cudaMemcpyAsync(&hs->err, h->d_err, sizeof(uint32_t), cudaMemcpyDeviceToHost, h->st), where));
    SG_TRY(check_cuda(cudaStreamSynchronize(h->st), where));
    SG_TRY(check_cuda(cudaGetLastError(), where));
    err = hs->err;
  } else {
    SG_TRY(check_cuda(cudaStreamSynchronize(h->st), where));
    SG_TRY(check_cuda(cudaGetLastError(), where));
    SG_TRY(check_cuda(cudaMemcpy(&err, h->d_err, sizeof(err), cudaMemcpyDeviceToHost), where));
  }
  if (err) {
    char buf[160];
    snprintf(buf, sizeof(buf), "%s: device check failed (flags 0x%x)", where, err);
    set_last_error(buf);
    return (err & kErrCsr) ? SPGEMM_ERR_INVALID_CSR : SPGEMM_ERR_DEVICE;
  }
  return SPGEMM_OK;
}

// Device time per phase: a pair of events around each timed region, read out (and the
// stream synchronised) only by spgemm_get_phase_times, so timing adds no synchronisation.
struct PhaseTimer {
  spgemm_ctx* h;
  int slot;
  cudaEvent_t a{};
  cudaStream_t st;
  PhaseTimer(spgemm_ctx* hh, int s, cudaStream_t stream = nullptr) : h(hh), slot(s), st(stream ? stream : hh->st) {
    if (!h->timing) return;
    cudaEventCreate(&a);
    cudaEventRecord(a, st);
  }
  void cancel() {
    if (!h->timing || !a) return;
    cudaEventDestroy(a);
    a = nullptr;
  }
  ~PhaseTimer() {
    if (!h->timing || !a) return;
    cudaEvent_t b;
    cudaEventCreate(&b);
    cudaEventRecord(b, st);
    h->timed[slot].push_back({a, b});
  }
};

void drain_timers(spgemm_ctx* h) {
  if (!h->timing) return;
  cudaStreamSynchronize(h->st);
  for (int s = 0; s < kPhaseSlots; ++s) {
    for (auto& pr : h->timed[s]) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, pr.first, pr.second) == cudaSuccess) h->phase_ms[s] += ms;
      h->phase_n[s] += 1;
      cudaEventDestroy(pr.first);
      cudaEventDestroy(pr.second);
    }
    h->timed[s].clear();
  }
}

int valid_csr_desc(const spgemm_csr* M, int64_t rows, int64_t cols) {
  if (!M) return 0;
  if (M->rows != rows || M->cols != cols || M->nnz < 0) return 0;
  if (!M->row_ptr) return 0;
  if (M->nnz > 0 && (!M->col_idx || !M->vals)) return 0;
  return 1;
}

// ---------------------------------------------------------------------------------------------
// Level-0 histogram of a batch, filled by the outer product (none when one chunk covers a row).
int alloc_counts0(spgemm_ctx* h, const HeavyBatch& hb, unsigned long long** out) {
  *out = nullptr;
  if (h->plan.chunks_required == 1) return SPGEMM_OK;
  const int64_t n = (hb.h1 - hb.h0) * h->plan.v_chunks[0];
  unsigned long long* c;
  SG_ALLOC(c, unsigned long long, n);
  cudaMemsetAsync(c, 0, sizeof(unsigned long long) * n, h->st);
  *out = c;
  return SPGEMM_OK;
}

// Heavy batch: expansion (MaskedCsr2Csc + OuterProduct of Algorithm 3).
int heavy_expand(spgemm_ctx* h, HeavyBatch& hb, bool vals, int64_t* c_rowptr, unsigned long long* counts0) {
  std::unique_ptr<PhaseTimer> tcsc(new PhaseTimer(h, 2));
  const int64_t R = hb.h1 - hb.h0;
  const int32_t* rows = h->d_heavy + hb.h0;
  const int64_t kc = h->k;
  int32_t* colcnt;
  int64_t *colptr, *slice_off;
  SG_ALLOC(colcnt, int32_t, kc);
  SG_ALLOC(colptr, int64_t, kc + 1);
  SG_ALLOC(slice_off, int64_t, kc + 1);
  cudaMemsetAsync(colcnt, 0, sizeof(int32_t) * kc, h->st);
  launch_csc_count(h->A, rows, R, colcnt, h->st);
  launch_slice_sizes(colcnt, h->B, kc, colptr, slice_off, h->st);
  SG_TRY(scan(h, colptr, colptr, kc));
  SG_TRY(scan(h, slice_off, slice_off, kc));
  // nnz of the masked A: sum of the heavy rows' lengths; bounded by nnz(A)
  int64_t nnzh = 0;
  SG_TRY(check_cuda(cudaMemcpyAsync(&nnzh, colptr + kc, sizeof(int64_t), cudaMemcpyDeviceToHost, h->st),
                    "copy masked nnz"));
  SG_TRY(check_cuda(cudaStreamSynchronize(h->st), "masked csc"));
  int32_t *csc_row, *csc_col;
  double* csc_val;
  int64_t* cursor;
  SG_ALLOC(csc_row, int32_t, nnzh);
  SG_ALLOC(csc_val, double, nnzh);
  SG_ALLOC(csc_col, int32_t, nnzh);
  SG_ALLOC(cursor, int64_t, std::max<int64_t>(kc, R));
  launch_copy_i64(colptr, cursor, kc, h->st);
  launch_csc_scatter(h->A, rows, R, cursor, csc_row, csc_val, csc_col, h->st);
  // C^ row pointers: heavy IP prefix of the batch; the cursor starts at each row's first slot
  launch_offset_copy(h->d_heavy_pre + hb.h0, R + 1, h->heavy_pre[hb.h0], c_rowptr, h->st);
  launch_copy_i64(c_rowptr, cursor, R, h->st);
  tcsc.reset();
  int2* part;
  SG_ALLOC(part, int2, std::max<int64_t>(1, ceil_div(hb.elems, kOpTile)));
  launch_partition(slice_off, kc, hb.elems, kOpTile, part, h->st);
  const spgemm_plan& P = h->plan;
  const int shift0 = ilog2_i64(P.chunk_width * P.chunks_required / P.v_chunks[0]);
  const int64_t v0 = P.v_chunks[0];
  unsigned long long* op_counts = counts0;
  // (bounded memory: the per-B-row counts take k * v0 int32; beyond 8 GB count per product)
  if (counts0 && !(h->opt.flags & SPGEMM_FLAG_FUSED_HIST) && kc * v0 <= (int64_t(1) << 31)) {
    // Level-0 histogram by factorisation: the products of A[r, k] fall in the chunks that row k
    // of B touches, so counts0[r, c] = sum over the entries (r, k) of (entries of B row k in
    // chunk c).  Per-B-row chunk counts, then one coalesced read per entry of A: work in the
    // entries of A and B instead of in the products.
    PhaseTimer t(h, 4);
    int32_t* bh;
    int64_t* hrp;
    SG_ALLOC(bh, int32_t, kc * v0);
    SG_ALLOC(hrp, int64_t, R + 1);
    cudaMemsetAsync(bh, 0, sizeof(int32_t) * kc * v0, h->st);
    launch_b_chunk_hist(h->B, colcnt, shift0, v0, bh, h->d_err, h->st);
    launch_heavy_row_len(h->A, rows, R, hrp, h->st);
    SG_TRY(scan(h, hrp, hrp, R));
    launch_row_chunk_counts(h->A, rows, R, hrp, nnzh, bh, v0, counts0, h->st);
    ws_free(h, bh);
    ws_free(h, hrp);
    op_counts = nullptr;
  }
  {
    PhaseTimer t(h, 3);
    launch_outer_product(colptr, csc_row, csc_val, csc_col, slice_off, part, hb.elems, h->B, cursor, h->d_chat_col,
                         vals ? h->d_chat_val : nullptr, vals, op_counts, shift0, v0, h->d_err, h->st);
  }
  ws_free(h, part);
  ws_free(h, colcnt);
  ws_free(h, colptr);
  ws_free(h, slice_off);
  ws_free(h, csc_row);
  ws_free(h, csc_val);
  ws_free(h, csc_col);
  ws_free(h, cursor);
  return SPGEMM_OK;
}

// Heavy batch: hierarchical multisplit (the reorder loop of Algorithm 3).  The symbolic pass records
// the level structure (which needs the heavy-chunk counts on the host); the numeric pass of a
// recomputed batch replays it without synchronising.
int heavy_levels(spgemm_ctx* h, HeavyBatch& hb, bool vals, bool record, const int64_t* c_rowptr,
                 unsigned long long* counts0) {
  const spgemm_plan& P = h->plan;
  const int64_t R = hb.h1 - hb.h0;
  const int64_t cap = h->batch_cap;
  if (record) hb.lv.clear();
  if (P.chunks_required == 1) {
    // one chunk per row: the rows of C^ are the final chunks
    if (record) {
      hb.nfinal = R;
      SG_ALLOC(hb.f_start, int64_t, R);
      SG_ALLOC(hb.f_cnt, int64_t, R);
      SG_ALLOC(hb.f_row, int32_t, R);
      SG_ALLOC(hb.f_base, int32_t, R);
      launch_final_desc(c_rowptr, 0, R, 0, nullptr, nullptr, hb.f_start, hb.f_cnt, hb.f_row, hb.f_base, h->st);
      hb.bitmap_from = 0;
    }
    return SPGEMM_OK;
  }
  // level inputs
  int64_t nin = R;
  const int64_t* in_ptr = c_rowptr;
  int64_t in_half = 0;  // which half of the C^ buffer holds the input
  int32_t* in_row = nullptr;
  int32_t* in_base = nullptr;
  int64_t in_width = P.chunk_width * P.chunks_required;  // padded column range of a C^ row
  int64_t* prev_ptr = nullptr;
  int64_t total_in = hb.elems;
  std::vector<void*> to_free;
  if (record) {
    // descriptor capacity: level l writes at most nin_l * v_l final chunks, and the next
    // level's input holds only heavy chunks (more than tau elements each)
    int64_t capd = 0, rows = R;
    for (int l = 0; l < P.levels; ++l) {
      capd += rows * P.v_chunks[l];
      rows = std::min<int64_t>(rows * P.v_chunks[l], hb.elems / (P.tau + 1));
    }
    hb.nfinal = 0;
    SG_ALLOC(hb.f_start, int64_t, capd);
    SG_ALLOC(hb.f_cnt, int64_t, capd);
    SG_ALLOC(hb.f_row, int32_t, capd);
    SG_ALLOC(hb.f_base, int32_t, capd);
  }
  for (int l = 0; l < P.levels; ++l) {
    const int64_t v = P.v_chunks[l];
    const int64_t width = in_width / v;
    const int shift = ilog2_i64(width);
    const bool last = (l == P.levels - 1);
    const int64_t nout = nin * v;
    LevelInfo li;
    if (record) {
      li.nin = nin;
      li.v = v;
      li.width = width;
      li.desc0 = hb.nfinal;
    } else {
      li = hb.lv[l];
    }
    unsigned long long* counts;
    int32_t *xmap = nullptr, *out_row, *out_base;
    int64_t* rptr;
    const bool fused = (l == 0 && counts0 != nullptr);  // level-0 counts came from the outer product
    if (fused) counts = counts0;
    else SG_ALLOC(counts, unsigned long long, nout);
    SG_ALLOC(rptr, int64_t, nout + 1);
    SG_ALLOC(out_row, int32_t, nout);
    SG_ALLOC(out_base, int32_t, nout);
    if (!fused) cudaMemsetAsync(counts, 0, sizeof(unsigned long long) * nout, h->st);
    const int32_t* in_col = h->d_chat_col + in_half * cap;
    const double* in_val = h->d_chat_val ? h->d_chat_val + in_half * cap : nullptr;
    const bool match = !(h->opt.flags & SPGEMM_FLAG_NO_MATCH);
    int2* part;
    SG_ALLOC(part, int2, std::max<int64_t>(1, ceil_div(total_in, kMsTile)));
    launch_partition(in_ptr, nin, total_in, kMsTile, part, h->st);
    if (!fused) {
      PhaseTimer t(h, 4);
      launch_histogram(in_ptr, part, total_in, in_col, shift, v, P.group_rows, counts, false, h->sms, h->d_err,
                       h->st);
    }
    if (!last) {
      // ThreshPartition of the chunks: heavy (count > tau) first, stable
      uint8_t* pbin;
      int32_t* plist;
      int64_t* pcnt;
      const int64_t nblk = bin_blocks(nout);
      SG_ALLOC(pbin, uint8_t, nout);
      SG_ALLOC(plist, int32_t, nout);
      SG_ALLOC(pcnt, int64_t, 2 * nblk + 1);
      SG_ALLOC(xmap, int32_t, nout);
      launch_chunk_partition(counts, nout, P.tau, pbin, h->st);
      launch_bin_count(pbin, nout, 2, pcnt, h->st);
      SG_TRY(scan(h, pcnt, pcnt, 2 * nblk));
      launch_bin_scatter(pbin, nout, 2, pcnt, plist, h->st);
      launch_invert(plist, nout, xmap, h->st);
      if (record) {
        int64_t nh = 0;
        SG_TRY(check_cuda(cudaMemcpyAsync(&nh, pcnt + nblk, sizeof(int64_t), cudaMemcpyDeviceToHost, h->st),
                          "copy heavy chunk count"));
        SG_TRY(check_cuda(cudaStreamSynchronize(h->st), "level partition"));
        li.nheavy = nh;
      }
      ws_free(h, pbin);
      ws_free(h, plist);
      ws_free(h, pcnt);
    } else {
      li.nheavy = 0;
    }
    {
      PhaseTimer t(h, 6);
      launch_reord_meta(counts, nin, v, xmap, in_row, in_base, width, rptr, out_row, out_base, h->st);
      SG_TRY(scan(h, rptr, rptr, nout));
    }
    // cursor for the multisplit reservations: starts at each C^_reord row's first slot
    unsigned long long* cursor;
    SG_ALLOC(cursor, unsigned long long, nout);
    launch_copy_i64(rptr, reinterpret_cast<int64_t*>(cursor), nout, h->st);
    const int64_t out_half = 1 - in_half;
    {
      PhaseTimer t(h, 5);
      const bool tma = (h->opt.flags & SPGEMM_FLAG_TMA_SPLIT) &&
                       launch_multisplit_tma(in_ptr, part, total_in, in_col, in_val, shift, v, P.group_rows, xmap,
                                             cursor, h->d_chat_col + out_half * cap,
                                             vals ? h->d_chat_val + out_half * cap : nullptr, vals, h->sms, h->d_err,
                                             h->st, static_cast<uint32_t>(std::max(0, h->opt.debug_wait_spins)));
      if (!tma)
        launch_multisplit(in_ptr, part, total_in, in_col, in_val, shift, v, P.group_rows, xmap, cursor,
                          h->d_chat_col + out_half * cap, vals ? h->d_chat_val + out_half * cap : nullptr, vals, match,
                          h->sms, h->d_err, h->st);
    }
    ws_free(h, part);
    ws_free(h, cursor);
    if (!fused) ws_free(h, counts);
    if (xmap) ws_free(h, xmap);
    // light outputs of this level (all outputs at the last level) are final chunks
    if (record) {
      const int64_t q0 = last ? 0 : li.nheavy;
      hb.bitmap_from = last ? hb.nfinal : hb.nfinal + (nout - q0);
      launch_final_desc(rptr, q0, nout, out_half * cap, out_row, out_base, hb.f_start + hb.nfinal,
                        hb.f_cnt + hb.nfinal, hb.f_row + hb.nfinal, hb.f_base + hb.nfinal, h->st);
      hb.nfinal += nout - q0;
      li.elem_base = out_half * cap;
      hb.lv.push_back(li);
    }
    // next level: the heavy chunks (stored first) of this level's output
    if (in_row) ws_free(h, in_row);
    if (in_base) ws_free(h, in_base);
    if (prev_ptr) ws_free(h, prev_ptr);
    if (last || li.nheavy == 0) {
      ws_free(h, rptr);
      ws_free(h, out_row);
      ws_free(h, out_base);
      break;
    }
    int64_t heavy_elems = 0;
    if (record) {
      SG_TRY(check_cuda(cudaMemcpyAsync(&heavy_elems, rptr + li.nheavy, sizeof(int64_t), cudaMemcpyDeviceToHost,
                                        h->st), "copy heavy chunk elements"));
      SG_TRY(check_cuda(cudaStreamSynchronize(h->st), "level input"));
      hb.lv.back().next_elems = heavy_elems;
    } else {
      heavy_elems = li.next_elems;
    }
    nin = li.nheavy;
    in_ptr = rptr;
    prev_ptr = rptr;
    in_row = out_row;
    in_base = out_base;
    in_half = out_half;
    in_width = width;
    total_in = heavy_elems;
  }
  return SPGEMM_OK;
}

// Chunk histogram of the rows of B that some heavy row uses (final chunk width): bh[k * v + c]
// = entries of row k in chunk c.  Computed once per handle and shared by every batch and both
// phases (the direct split of level 0 and the generated chunks read it).
int ensure_bh(spgemm_ctx* h) {
  if (h->d_bh) return SPGEMM_OK;
  const int64_t kc = h->k;
  const int64_t v = h->plan.chunks_required;
  SG_ALLOC(h->d_colcnt, int32_t, std::max<int64_t>(kc, 1));
  SG_ALLOC(h->d_bh, int32_t, std::max<int64_t>(kc * v, 1));
  cudaMemsetAsync(h->d_colcnt, 0, sizeof(int32_t) * kc, h->st);
  cudaMemsetAsync(h->d_bh, 0, sizeof(int32_t) * kc * v, h->st);
  launch_csc_count(h->A, h->d_heavy, h->nheavy, h->d_colcnt, h->st);
  launch_b_chunk_hist(h->B, h->d_colcnt, ilog2_i64(h->plan.chunk_width), v, h->d_bh, h->d_err, h->st);
  return SPGEMM_OK;
}

// Heavy batch, direct split (SPGEMM_FLAG_DIRECT_SPLIT, one-level plans): the per-(row, chunk)
// counts come from per-B-row chunk histograms, and the outer product writes every element straight
// into its C^_reord row, so C^ never reaches global memory and level 0 needs no multisplit pass.
int heavy_direct(spgemm_ctx* h, HeavyBatch& hb, bool vals, bool record) {
  const spgemm_plan& P = h->plan;
  const int64_t R = hb.h1 - hb.h0;
  const int32_t* rows = h->d_heavy + hb.h0;
  const int64_t kc = h->k;
  const int64_t v = P.v_chunks[0];
  const int64_t width = P.chunk_width;
  const int shift = ilog2_i64(width);
  std::unique_ptr<PhaseTimer> tcsc(new PhaseTimer(h, 2));
  int32_t* colcnt;
  int64_t *colptr, *slice_off;
  SG_ALLOC(colcnt, int32_t, kc);
  SG_ALLOC(colptr, int64_t, kc + 1);
  SG_ALLOC(slice_off, int64_t, kc + 1);
  cudaMemsetAsync(colcnt, 0, sizeof(int32_t) * kc, h->st);
  launch_csc_count(h->A, rows, R, colcnt, h->st);
  launch_slice_sizes(colcnt, h->B, kc, colptr, slice_off, h->st);
  SG_TRY(scan(h, colptr, colptr, kc));
  SG_TRY(scan(h, slice_off, slice_off, kc));
  // A batch whose chunks the symbolic phase counted from generated products (the numeric
  // expansion of a recomputed batch) already knows its entries and, in its descriptors, where
  // every (row, chunk) run of C^_reord starts: no synchronisation and no second count.
  const bool from_symbolic = h->gen_symbolic && !record;
  int64_t nnzh = 0;
  if (from_symbolic) {
    nnzh = hb.entries;
  } else {
    SG_TRY(check_cuda(cudaMemcpyAsync(&nnzh, colptr + kc, sizeof(int64_t), cudaMemcpyDeviceToHost, h->st),
                      "copy masked nnz"));
    SG_TRY(check_cuda(cudaStreamSynchronize(h->st), "masked csc"));
  }
  int32_t *csc_row, *csc_col;
  double* csc_val;
  int64_t* cursor;
  SG_ALLOC(csc_row, int32_t, nnzh);
  SG_ALLOC(csc_val, double, nnzh);
  SG_ALLOC(csc_col, int32_t, nnzh);
  SG_ALLOC(cursor, int64_t, std::max<int64_t>(kc, R * v));
  launch_copy_i64(colptr, cursor, kc, h->st);
  launch_csc_scatter(h->A, rows, R, cursor, csc_row, csc_val, csc_col, h->st);
  unsigned long long* counts = nullptr;
  int64_t* rptr = nullptr;
  int32_t *out_row = nullptr, *out_base = nullptr;
  const int64_t nout = R * v;
  if (from_symbolic) {
    launch_cursor_from_desc(hb.f_start, hb.f_row, hb.f_base, hb.nfinal, v, shift, cursor, h->st);
  } else {
    // level-0 histogram from the chunk histograms of the rows of B
    int32_t* bh;
    SG_TRY(ensure_bh(h));
    bh = h->d_bh;
    SG_ALLOC(counts, unsigned long long, nout);
    SG_ALLOC(rptr, int64_t, nout + 1);
    SG_ALLOC(out_row, int32_t, nout);
    SG_ALLOC(out_base, int32_t, nout);
    int64_t* hrp;
    SG_ALLOC(hrp, int64_t, R + 1);
    cudaMemsetAsync(counts, 0, sizeof(unsigned long long) * nout, h->st);
    launch_heavy_row_len(h->A, rows, R, hrp, h->st);
    SG_TRY(scan(h, hrp, hrp, R));
    launch_row_chunk_counts(h->A, rows, R, hrp, nnzh, bh, v, counts, h->st);
    ws_free(h, hrp);
    launch_reord_meta(counts, R, v, nullptr, nullptr, nullptr, width, rptr, out_row, out_base, h->st);
    SG_TRY(scan(h, rptr, rptr, nout));
    launch_copy_i64(rptr, cursor, nout, h->st);
  }
  OdTile* part;
  SG_ALLOC(part, OdTile, std::max<int64_t>(1, ceil_div(hb.elems, kOdTile)));
  launch_od_partition(slice_off, kc, hb.elems, colptr, h->B, part, h->st);
  tcsc.reset();
  {
    PhaseTimer t(h, 3);
    launch_outer_direct(colptr, csc_row, csc_val, csc_col, slice_off, part, hb.elems, h->B,
                        reinterpret_cast<unsigned long long*>(cursor), h->d_chat_col,
                        vals ? h->d_chat_val : nullptr, vals, shift, v, h->d_err, h->st);
  }
  if (record) {
    hb.lv.clear();
    LevelInfo li;
    li.nin = R;
    li.v = v;
    li.width = width;
    li.nheavy = 0;
    li.desc0 = 0;
    li.elem_base = 0;
    hb.lv.push_back(li);
    hb.nfinal = nout;
    hb.bitmap_from = 0;
    SG_ALLOC(hb.f_start, int64_t, nout);
    SG_ALLOC(hb.f_cnt, int64_t, nout);
    SG_ALLOC(hb.f_row, int32_t, nout);
    SG_ALLOC(hb.f_base, int32_t, nout);
    launch_final_desc(rptr, 0, nout, 0, out_row, out_base, hb.f_start, hb.f_cnt, hb.f_row, hb.f_base, h->st);
  }
  for (void* p : {static_cast<void*>(colcnt), static_cast<void*>(colptr), static_cast<void*>(slice_off),
                  static_cast<void*>(csc_row), static_cast<void*>(csc_val), static_cast<void*>(csc_col),
                  static_cast<void*>(cursor),
                  static_cast<void*>(counts), static_cast<void*>(rptr),
                  static_cast<void*>(out_row), static_cast<void*>(out_base), static_cast<void*>(part)})
    ws_free(h, p);
  return SPGEMM_OK;
}

// One-level plans split level 0 inside the outer product (products written at their reserved
// C^_reord positions, counts from the per-B-row chunk histograms), unless the caller asks for the
// separate multisplit pass (SPGEMM_FLAG_EXPAND_SPLIT) or for one of its variants (plain atomics,
// bulk-copy tiles, the per-product histogram).  Measured on GB300: R-MAT scale 21 4.33 s against
// 5.26 s per product, the Markov-clustering expansion 531 against 625 ms.
bool use_direct(const spgemm_ctx* h) {
  const int separate = SPGEMM_FLAG_EXPAND_SPLIT | SPGEMM_FLAG_NO_MATCH | SPGEMM_FLAG_TMA_SPLIT | SPGEMM_FLAG_FUSED_HIST;
  return !(h->opt.flags & separate) && h->plan.levels == 1 && h->plan.chunks_required > 1;
}

// ---- heavy rows without C^ (SPGEMM_FLAG_FUSED) ------------------------------------------------
FusedSrc fused_src(const spgemm_ctx* h, const HeavyBatch& hb, const int32_t* seg) {
  FusedSrc f{};
  f.arp = h->A.row_ptr;
  f.aval = h->A.vals;
  f.hrp = hb.f_hrp;
  f.seg = seg;
  f.E = hb.entries;
  f.bcol = h->d_bs_col;
  f.bval = h->d_bs_val;
  f.shift = ilog2_i64(h->plan.chunk_width);
  return f;
}

// The batch's segment table (built from the current split of B), for one phase's chunk kernels.
// One buffer on the handle, grown to the largest batch during the symbolic phase, so the numeric
// phase allocates nothing (and can be captured into a graph).
int fused_segtable(spgemm_ctx* h, const HeavyBatch& hb, int32_t** seg) {
  const int64_t v = h->plan.chunks_required;
  const int64_t need = std::max<int64_t>((v + 1) * hb.entries, 1);
  if (need > h->seg_cap) {
    ws_free(h, h->d_seg);
    h->d_seg = nullptr;
    h->seg_cap = 0;
    SG_ALLOC(h->d_seg, int32_t, need);
    h->seg_cap = need;
  }
  if (hb.entries > h->ecol_cap) {
    ws_free(h, h->d_ecol);
    h->d_ecol = nullptr;
    h->ecol_cap = 0;
    SG_ALLOC(h->d_ecol, int32_t, std::max<int64_t>(hb.entries, 1));
    h->ecol_cap = hb.entries;
  }
  *seg = h->d_seg;
  launch_segtable(h->A, h->d_heavy + hb.h0, hb.h1 - hb.h0, hb.f_hrp, h->B, h->d_bo, v, hb.entries, h->d_ecol, *seg,
                  h->st);
  return SPGEMM_OK;
}

// The column split of B (the multisplit applied to B's rows by the final chunk width): the
// symbolic phase counts the chunk entries of every row of B that a heavy row uses and splits
// the columns; the numeric phase splits columns and values again (A and B may have new values).
int fused_prepare(spgemm_ctx* h, bool vals) {
  PhaseTimer t(h, 2);
  const int64_t kc = h->k;
  const int64_t v = h->plan.chunks_required;
  const int shift = ilog2_i64(h->plan.chunk_width);
  SG_TRY(ensure_bh(h));
  if (!h->d_bo) {
    SG_ALLOC(h->d_bo, int32_t, std::max<int64_t>(kc * (v + 1), 1));
    SG_ALLOC(h->d_bs_col, int32_t, std::max<int64_t>(h->B.nnz, 1));
  }
  if (vals && !h->d_bs_val) SG_ALLOC(h->d_bs_val, double, std::max<int64_t>(h->B.nnz, 1));
  launch_bsplit(h->B, h->d_colcnt, h->d_bh, shift, v, h->d_bo, h->d_bs_col, vals ? h->d_bs_val : nullptr, h->d_err,
                h->st);
  return SPGEMM_OK;
}

// Final chunks of a batch: the level-0 counts from the per-B-row chunk counts, one final chunk
// per (row, chunk), chunk-major.  Symbolic phase only; the numeric phase reuses them.
int heavy_fused(spgemm_ctx* h, HeavyBatch& hb) {
  const int64_t R = hb.h1 - hb.h0;
  const int32_t* rows = h->d_heavy + hb.h0;
  const int64_t v = h->plan.chunks_required;
  const int64_t W = h->plan.chunk_width;
  PhaseTimer t(h, 4);
  int64_t*& hrp = hb.f_hrp;
  unsigned long long* counts;
  SG_ALLOC(hrp, int64_t, R + 1);
  SG_ALLOC(counts, unsigned long long, R * v);
  launch_heavy_row_len(h->A, rows, R, hrp, h->st);
  SG_TRY(scan(h, hrp, hrp, R));
  SG_TRY(check_cuda(cudaMemcpyAsync(&hb.entries, hrp + R, sizeof(int64_t), cudaMemcpyDeviceToHost, h->st),
                    "copy heavy entries"));
  cudaMemsetAsync(counts, 0, sizeof(unsigned long long) * R * v, h->st);
  SG_TRY(check_cuda(cudaStreamSynchronize(h->st), "heavy entries"));
  const int64_t entries = hb.entries;
  launch_row_chunk_counts(h->A, rows, R, hrp, entries, h->d_bh, v, counts, h->st);
  hb.lv.clear();
  LevelInfo li;
  li.nin = R;
  li.v = v;
  li.width = W;
  hb.lv.push_back(li);
  hb.nfinal = R * v;
  hb.bitmap_from = 0;
  SG_ALLOC(hb.f_start, int64_t, R * v);
  SG_ALLOC(hb.f_cnt, int64_t, R * v);
  SG_ALLOC(hb.f_row, int32_t, R * v);
  SG_ALLOC(hb.f_base, int32_t, R * v);
  int64_t* rptr = nullptr;
  if (h->gen_symbolic) {  // where every (row, chunk) run of the numeric expansion starts
    SG_ALLOC(rptr, int64_t, R * v + 1);
    SG_TRY(scan(h, reinterpret_cast<const int64_t*>(counts), rptr, R * v));
  }
  launch_fused_desc(counts, rptr, R, v, W, hb.f_cnt, hb.f_row, hb.f_base, hb.f_start, h->st);
  ws_free(h, counts);
  ws_free(h, rptr);
  return SPGEMM_OK;
}

// Accumulator bins of the final chunks (stable order), then their symbolic counts and the
// offsets of every chunk inside its row of C.
int heavy_chunk_symbolic(spgemm_ctx* h, HeavyBatch& hb, int64_t* row_nnz) {
  const int64_t nf = hb.nfinal;
  const int64_t R = hb.h1 - hb.h0;
  const int nb = h->lad.n + 4;  // chunk bins: hash ladder + 4 bitmap bins
  SG_ALLOC(hb.f_nnz, int64_t, nf);
  SG_ALLOC(hb.f_out, int64_t, nf);
  SG_ALLOC(hb.f_list, int32_t, nf);
  cudaMemsetAsync(hb.f_nnz, 0, sizeof(int64_t) * nf, h->st);
  {
    uint8_t* fbin;
    int64_t* fcnt;
    int64_t* starts;
    const int64_t nblk = bin_blocks(nf);
    SG_ALLOC(fbin, uint8_t, nf);
    SG_ALLOC(fcnt, int64_t, nb * nblk + 1);
    SG_ALLOC(starts, int64_t, nb + 1);
    launch_chunk_classify(hb.f_cnt, nf, hb.bitmap_from, h->rule, fbin, h->st);
    launch_bin_count(fbin, nf, nb, fcnt, h->st);
    SG_TRY(scan(h, fcnt, fcnt, nb * nblk));
    launch_bin_scatter(fbin, nf, nb, fcnt, hb.f_list, h->st);
    launch_bin_starts(fcnt, nblk, nb, starts, h->st);
    hb.f_bin_start.assign(nb + 1, 0);
    SG_TRY(check_cuda(cudaMemcpyAsync(hb.f_bin_start.data(), starts, sizeof(int64_t) * (nb + 1),
                                      cudaMemcpyDeviceToHost, h->st), "copy chunk bins"));
    SG_TRY(check_cuda(cudaStreamSynchronize(h->st), "chunk bins"));
    ws_free(h, fbin);
    ws_free(h, fcnt);
    ws_free(h, starts);
  }
  if (!h->fused && !(h->opt.flags & SPGEMM_FLAG_HASH_PER_CHUNK)) {
    // descriptors of the two numeric hash bins: one buffer sized by the largest batch, so the
    // numeric phase allocates nothing
    const int b0 = h->lad.n;
    const int64_t need = hb.f_bin_start[b0 + 2] - hb.f_bin_start[b0];  // the two hash bins
    if (need > h->cdesc_cap) {
      ws_free(h, h->d_cdesc);
      h->d_cdesc = nullptr;
      h->cdesc_cap = 0;
      SG_ALLOC(h->d_cdesc, ChunkDesc, need);
      h->cdesc_cap = need;
    }
  }
  int32_t* seg = nullptr;
  const bool gen = h->fused || h->gen_symbolic;  // the chunks' products are generated
  {
    PhaseTimer t(h, 7);
    if (gen) SG_TRY(fused_segtable(h, hb, &seg));
    ChunkSet cs{};
    cs.start = hb.f_start;
    cs.cnt = hb.f_cnt;
    cs.row = hb.f_row;
    cs.base = hb.f_base;
    cs.nnz = hb.f_nnz;
    cs.heavy_rows = h->d_heavy + hb.h0;
    cs.col = h->d_chat_col;
    cs.val = nullptr;
    Sink sk{};
    sk.row_begin = 0;
    sk.row_end = h->m;
    for (int L = 0; L < h->lad.n; ++L)  // light chunks of early levels: hash ladder
      launch_chunks(cs, hb.f_list + hb.f_bin_start[L], hb.f_bin_start[L + 1] - hb.f_bin_start[L],
                    h->lad.slots[L], h->lad.tpr[L], false, 0, false, sk, h->d_err, h->st);
    for (int j = 0; j < 4; ++j) {        // last-level chunks: bitmaps of width W
      const int b = h->lad.n + j;
      if (gen)
        launch_fused_chunks(fused_src(h, hb, seg), cs, hb.f_list + hb.f_bin_start[b],
                            hb.f_bin_start[b + 1] - hb.f_bin_start[b], h->plan.chunk_width, 0, 0, kFusedSymTpr[j], sk,
                            h->d_err, h->d_counter, h->st);
      else
        launch_chunk_bitmap(cs, hb.f_list + hb.f_bin_start[b], hb.f_bin_start[b + 1] - hb.f_bin_start[b],
                            h->plan.chunk_width, 0, 0, kChunkSymTpr[j], sk, h->d_err, h->d_counter, nullptr, h->st);
    }
  }
  {
    // element and nnz totals of the dense-accumulator chunks (for the statistics)
    const int bd = h->lad.n + 3;
    unsigned long long* sums;
    SG_ALLOC(sums, unsigned long long, 2);
    cudaMemsetAsync(sums, 0, 2 * sizeof(unsigned long long), h->st);
    launch_list_sums(hb.f_list + hb.f_bin_start[bd], hb.f_bin_start[bd + 1] - hb.f_bin_start[bd], hb.f_cnt,
                     hb.f_nnz, sums, h->st);
    SG_TRY(check_cuda(cudaMemcpyAsync(hb.dense_sums, sums, 2 * sizeof(int64_t), cudaMemcpyDeviceToHost, h->st),
                      "copy dense sums"));
    ws_free(h, sums);
  }
  // offsets of the chunks inside their rows
  PhaseTimer toff(h, 8);
  const int64_t nfin = h->plan.chunks_required;
  const int shift_fin = ilog2_i64(h->plan.chunk_width);
  int64_t* grid;
  SG_ALLOC(grid, int64_t, R * nfin + 1);
  cudaMemsetAsync(grid, 0, sizeof(int64_t) * (R * nfin + 1), h->st);
  launch_grid_fill(hb.f_row, hb.f_base, hb.f_nnz, nf, shift_fin, nfin, grid, h->st);
  SG_TRY(scan(h, grid, grid, R * nfin));
  launch_grid_finish(grid, hb.f_row, hb.f_base, nf, shift_fin, nfin, hb.f_out, h->st);
  launch_row_totals(grid, R, nfin, h->d_heavy + hb.h0, row_nnz, h->st);
  SG_TRY(check_cuda(cudaMemcpyAsync(&hb.nnz_c, grid + R * nfin, sizeof(int64_t), cudaMemcpyDeviceToHost, h->st),
                    "copy heavy nnz"));
  ws_free(h, grid);
  return SPGEMM_OK;
}

int heavy_chunk_numeric(spgemm_ctx* h, HeavyBatch& hb, const Sink& sk) {
  PhaseTimer t(h, 11);
  int32_t* seg = nullptr;
  if (h->fused) SG_TRY(fused_segtable(h, hb, &seg));
  ChunkSet cs{};
  cs.start = hb.f_start;
  cs.cnt = hb.f_cnt;
  cs.row = hb.f_row;
  cs.base = hb.f_base;
  cs.nnz = hb.f_nnz;
  cs.out = hb.f_out;
  cs.heavy_rows = h->d_heavy + hb.h0;
  cs.col = h->d_chat_col;
  cs.val = h->d_chat_val;
  for (int L = 0; L < h->lad.n; ++L)
    launch_chunks(cs, hb.f_list + hb.f_bin_start[L], hb.f_bin_start[L + 1] - hb.f_bin_start[L], h->lad.slots[L],
                  h->lad.tpr[L], false, 0, true, sk, h->d_err, h->st);
  if ((h->opt.flags & SPGEMM_FLAG_DENSE_L2) && !h->fused && !h->d_gacc)
    SG_ALLOC(h->d_gacc, double, static_cast<int64_t>(h->sms) * h->plan.chunk_width);
  for (int j = 0; j < 4; ++j) {
    const int b = h->lad.n + j;
    PhaseTimer td(h, 12);  // only the dense bin is counted here (its region nests in slot 11)
    if (j < 3) td.cancel();
    if (h->fused)
      launch_fused_chunks(fused_src(h, hb, seg), cs, hb.f_list + hb.f_bin_start[b],
                          hb.f_bin_start[b + 1] - hb.f_bin_start[b], h->plan.chunk_width, j == 3 ? 2 : 1,
                          kChunkSlots[j], kChunkTpr[j], sk, h->d_err, h->d_counter, h->st);
    else if (j < 2 && !(h->opt.flags & SPGEMM_FLAG_HASH_PER_CHUNK))
      launch_chunk_groups(cs, hb.f_list + hb.f_bin_start[b], hb.f_bin_start[b + 1] - hb.f_bin_start[b],
                          h->plan.chunk_width, j == 0, sk,
                          h->d_cdesc + (j == 0 ? 0 : hb.f_bin_start[b] - hb.f_bin_start[b - 1]), h->d_err, h->st);
    else
      launch_chunk_bitmap(cs, hb.f_list + hb.f_bin_start[b], hb.f_bin_start[b + 1] - hb.f_bin_start[b],
                          h->plan.chunk_width, j == 3 ? 2 : 1, kChunkSlots[j], kChunkTpr[j], sk, h->d_err,
                          h->d_counter, h->d_gacc, h->st);
  }
  return SPGEMM_OK;
}

int ensure_chat(spgemm_ctx* h, bool vals) {
  const int64_t halves = use_direct(h) ? 1 : 2;  // the multisplit's double buffer, or C^_reord alone
  if (!h->d_chat_col) SG_ALLOC(h->d_chat_col, int32_t, halves * h->batch_cap);
  if (vals && !h->d_chat_val) SG_ALLOC(h->d_chat_val, double, halves * h->batch_cap);
  return SPGEMM_OK;
}

// Light rows run on their own stream (the paper's light queue) so that they overlap the heavy
// pipeline on the handle's stream: fork after everything enqueued so far, join before the
// next dependent step.
void fork_light(spgemm_ctx* h) {
  cudaEventRecord(h->ev_fork, h->st);
  cudaStreamWaitEvent(h->st_light, h->ev_fork, 0);
}
void join_light(spgemm_ctx* h) {
  cudaEventRecord(h->ev_join, h->st_light);
  cudaStreamWaitEvent(h->st, h->ev_join, 0);
}

// Numeric bins of the light hash rows by their exact nnz, from the row_ptr of C.  Enqueued at the
// end of the symbolic phase with the bin starts copied into `starts` (page-locked) and read after
// that phase's synchronisation; `starts` null: a synchronous pass of its own.
int numeric_bins_enqueue(spgemm_ctx* h, const int64_t* c_row_ptr, int64_t* starts_host) {
  const int nl = h->lad.n;
  int64_t nh = 0;  // hash rows outside the ESC levels (those keep their IP lists)
  for (int L = h->esc_levels; L < nl; ++L) nh += h->bin_start[2 * L + 1] - h->bin_start[2 * L];
  if (nh == 0) {
    h->nbin_start.assign(nl + 1, 0);
    return SPGEMM_OK;
  }
  int32_t* all;
  uint8_t* bin;
  int64_t *cnt, *starts;
  const int64_t nblk = bin_blocks(nh);
  SG_ALLOC(all, int32_t, nh);
  SG_ALLOC(h->d_nrows, int32_t, nh);
  SG_ALLOC(bin, uint8_t, nh);
  SG_ALLOC(cnt, int64_t, nl * nblk + 1);
  SG_ALLOC(starts, int64_t, nl + 1);
  int64_t off = 0;
  for (int L = h->esc_levels; L < nl; ++L) {
    const int64_t c = h->bin_start[2 * L + 1] - h->bin_start[2 * L];
    if (c) cudaMemcpyAsync(all + off, h->d_rows + h->bin_start[2 * L], sizeof(int32_t) * c, cudaMemcpyDeviceToDevice,
                           h->st);
    off += c;
  }
  launch_nnz_bins(all, nh, c_row_ptr, h->rule, bin, h->st);
  launch_bin_count(bin, nh, nl, cnt, h->st);
  SG_TRY(scan(h, cnt, cnt, nl * nblk));
  // the scatter writes positions into the concatenated list; map them back to row ids
  launch_bin_scatter(bin, nh, nl, cnt, h->d_nrows, h->st);
  launch_gather_rows(all, h->d_nrows, nh, h->st);
  launch_bin_starts(cnt, nblk, nl, starts, h->st);
  if (starts_host) {
    SG_TRY(check_cuda(cudaMemcpyAsync(starts_host, starts, sizeof(int64_t) * (nl + 1), cudaMemcpyDeviceToHost,
                                      h->st), "copy numeric bins"));
  } else {
    h->nbin_start.assign(nl + 1, 0);
    SG_TRY(check_cuda(cudaMemcpyAsync(h->nbin_start.data(), starts, sizeof(int64_t) * (nl + 1),
                                      cudaMemcpyDeviceToHost, h->st), "copy numeric bins"));
    SG_TRY(check_cuda(cudaStreamSynchronize(h->st), "numeric bins"));
  }
  ws_free(h, all);
  ws_free(h, bin);
  ws_free(h, cnt);
  ws_free(h, starts);
  return SPGEMM_OK;
}

// Numeric bins, if the symbolic phase did not leave them (exact workflow only: the estimated
// workflows accumulate the light rows during the symbolic phase).
int numeric_bins(spgemm_ctx* h) {
  if (!h->nbin_start.empty() || h->workflow != SPGEMM_WORKFLOW_SYMBOLIC) return SPGEMM_OK;
  return numeric_bins_enqueue(h, h->c_row_ptr, nullptr);
}

void light_pass(spgemm_ctx* h, bool numeric, const Sink& sk) {
  for (int L = 0; L < h->lad.n; ++L) {
    for (int d = 0; d < 2; ++d) {
      const int b = 2 * L + d;
      // short hash rows (IP lists): expand-sort-compact in registers; short rows of narrow span
      // keep the shortened dense accumulator, which measured faster for them
      const bool esc = L < h->esc_levels && d == 0;
      if (esc)
        launch_esc(h->A, h->B, h->d_rows + h->bin_start[b], h->bin_start[b + 1] - h->bin_start[b], numeric, sk,
                   h->d_err, h->st_light);
      if (esc && !numeric) continue;  // numeric: the rows binned here by nnz still follow
      RowJob job;
      if (numeric && d == 0) {  // hash rows: numeric bins by exact size
        job.rows = h->d_nrows + h->nbin_start[L];
        job.count = h->nbin_start[L + 1] - h->nbin_start[L];
      } else {
        job.rows = h->d_rows + h->bin_start[b];
        job.count = h->bin_start[b + 1] - h->bin_start[b];
      }
      job.slots = h->lad.slots[L];
      job.tpr = h->lad.tpr[L];
      job.dense = d == 1;
      launch_light(h->A, h->B, h->d_span_lo, job, numeric, sk, h->d_err, h->st_light);
    }
  }
}

// ---- heavy rows by the long-row hash (SPGEMM_FLAG_LONG_ROWS) -----------------------------------
// The heavy rows in groups whose global tables fit a budget (a quarter of the free memory, at most
// 8 GB): table slots per row from its IP (symbolic) or its nnz (numeric), a bitmap of C's columns
// per block for the ordered write.  Numeric rows outside [sk.row_begin, sk.row_end) are skipped.
int long_pass(spgemm_ctx* h, bool numeric, const Sink& sk) {
  const int64_t R = h->nheavy;
  if (R == 0) return SPGEMM_OK;
  PhaseTimer t(h, numeric ? 11 : 7);
  int64_t* cap;
  SG_ALLOC(cap, int64_t, R + 1);
  launch_long_caps(h->d_heavy, R, h->d_ip, numeric ? h->c_row_ptr : nullptr, cap, h->st);
  SG_TRY(scan(h, cap, cap, R));
  std::vector<int64_t> pre(static_cast<size_t>(R + 1));
  SG_TRY(check_cuda(cudaMemcpyAsync(pre.data(), cap, sizeof(int64_t) * (R + 1), cudaMemcpyDeviceToHost, h->st),
                    "copy long-row tables"));
  SG_TRY(check_cuda(cudaStreamSynchronize(h->st), "long-row tables"));
  size_t fr = 0, tot = 0;
  cudaMemGetInfo(&fr, &tot);
  const int64_t slot_bytes = numeric ? 12 : 4;
  const int64_t budget = std::max<int64_t>(std::min<int64_t>(int64_t(8) << 30, static_cast<int64_t>(fr / 4)),
                                           (pre[1] - pre[0]) * slot_bytes);
  const int blocks = long_blocks(h->sms);
  const int64_t nwords = (h->n + 31) / 32;
  uint32_t* bits = nullptr;
  if (numeric) SG_ALLOC(bits, uint32_t, std::max<int64_t>(2 * nwords * blocks, 1));
  int64_t j0 = 0;
  while (j0 < R) {
    int64_t j1 = j0 + 1;  // at least one row, then as many as fit the budget
    while (j1 < R && (pre[j1 + 1] - pre[j0]) * slot_bytes <= budget) ++j1;
    const int64_t slots = pre[j1] - pre[j0];
    int32_t* gkeys;
    double* gvals = nullptr;
    SG_ALLOC(gkeys, int32_t, slots);
    if (numeric) SG_ALLOC(gvals, double, slots);
    launch_long(h->A, h->B, h->d_heavy + j0, j1 - j0, cap + j0, pre[j0], gkeys, gvals, bits, nwords, numeric, sk,
                blocks, h->d_err, h->st);
    ws_free(h, gkeys);
    if (gvals) ws_free(h, gvals);
    j0 = j1;
  }
  if (bits) ws_free(h, bits);
  ws_free(h, cap);
  return SPGEMM_OK;
}

// ---- estimated light-row sizing (Ocean page: Table 1, the estimation-based workflow) -------

// Stable split of a row list by a per-item bin in [0, nb): `out` receives the rows bin by bin,
// `starts` (host, nb + 1) the bin boundaries.  Synchronises to read them.
int split_rows(spgemm_ctx* h, const int32_t* rows, int64_t n, const uint8_t* bin, int nb, int32_t* out,
               std::vector<int64_t>& starts) {
  starts.assign(nb + 1, 0);
  if (n == 0) return SPGEMM_OK;
  const int64_t nblk = bin_blocks(n);
  int64_t *cnt, *st;
  SG_ALLOC(cnt, int64_t, nb * nblk + 1);
  SG_ALLOC(st, int64_t, nb + 1);
  launch_bin_count(bin, n, nb, cnt, h->st);
  SG_TRY(scan(h, cnt, cnt, nb * nblk));
  launch_bin_scatter(bin, n, nb, cnt, out, h->st);  // item index at its position
  launch_gather_rows(rows, out, n, h->st);           // item index -> row id
  launch_bin_starts(cnt, nblk, nb, st, h->st);
  SG_TRY(check_cuda(cudaMemcpyAsync(starts.data(), st, sizeof(int64_t) * (nb + 1), cudaMemcpyDeviceToHost, h->st),
                    "copy split"));
  SG_TRY(check_cuda(cudaStreamSynchronize(h->st), "split"));
  ws_free(h, cnt);
  ws_free(h, st);
  return SPGEMM_OK;
}

int ensure_sketch(spgemm_ctx* h) {
  if (h->d_sketch) return SPGEMM_OK;
  SG_ALLOC(h->d_sketch, uint8_t, std::max<int64_t>(h->B.rows, 1) * h->hll_m);
  launch_hll_sketch(h->B, h->hll_m, h->d_sketch, h->st);
  return SPGEMM_OK;
}

// The workflow of the light rows (Table 1 of the Ocean page for SPGEMM_WORKFLOW_AUTO): the
// upper bound when the average row has fewer than 64 products; HyperLogLog estimates when the
// expansion ratio (products per entry of A) and the compression ratio (products per entry of
// C) of a row sample -- 3% of the light rows, at least 600 and at most 10,000, evenly spaced --
// are both at least 8; else the exact symbolic pass.  The sample holds light rows only: the
// workflow sizes only those, and a heavy row's sketch merge would be one warp's long serial
// loop.
int choose_workflow(spgemm_ctx* h) {
  const int64_t ipt = h->stats.ip_total;
  const double er = h->A.nnz > 0 ? static_cast<double>(ipt) / static_cast<double>(h->A.nnz) : 0.0;
  h->hll_m = h->opt.hll_registers ? h->opt.hll_registers : (er < 48.0 ? 32 : 64);
  h->hll_coef = h->opt.hll_coef > 0.0 ? h->opt.hll_coef : (h->hll_m == 32 ? 2.0 : 1.5);
  int wf = h->opt.workflow;
  if (wf == SPGEMM_WORKFLOW_AUTO) {
    if (h->m > 0 && static_cast<double>(ipt) / static_cast<double>(h->m) < 64.0) {
      wf = SPGEMM_WORKFLOW_UPPER_BOUND;
    } else if (er < 8.0) {
      wf = SPGEMM_WORKFLOW_SYMBOLIC;
    } else if (h->bin_start[2 * h->lad.n] > 0) {
      const int64_t nlight = h->bin_start[2 * h->lad.n];  // d_rows[0, nlight): the light rows
      const int64_t want = std::min<int64_t>(
          nlight, std::max<int64_t>(600, std::min<int64_t>(10000, (3 * nlight + 50) / 100)));
      std::vector<int32_t> rows(want);  // positions in the light list, then row ids
      for (int64_t j = 0; j < want; ++j) rows[j] = static_cast<int32_t>(j * nlight / want);
      int32_t* d_rows;
      int64_t *d_ipv, *d_capv;
      double* d_est;
      SG_ALLOC(d_rows, int32_t, want);
      SG_ALLOC(d_ipv, int64_t, want);
      SG_ALLOC(d_capv, int64_t, h->m);
      SG_ALLOC(d_est, double, want);
      SG_TRY(check_cuda(cudaMemcpyAsync(d_rows, rows.data(), sizeof(int32_t) * want, cudaMemcpyHostToDevice, h->st),
                        "copy sample"));
      launch_gather_rows(h->d_rows, d_rows, want, h->st);
      SG_TRY(ensure_sketch(h));
      launch_hll_rows(h->A, d_rows, want, h->d_ip, h->d_sketch, h->hll_m, h->hll_coef, d_capv, d_est, h->st);
      launch_gather_ip(d_rows, want, h->d_ip, d_ipv, h->st);
      std::vector<double> est(want);
      std::vector<int64_t> ipv(want);
      SG_TRY(check_cuda(cudaMemcpyAsync(est.data(), d_est, sizeof(double) * want, cudaMemcpyDeviceToHost, h->st),
                        "copy sample estimates"));
      SG_TRY(check_cuda(cudaMemcpyAsync(ipv.data(), d_ipv, sizeof(int64_t) * want, cudaMemcpyDeviceToHost, h->st),
                        "copy sample products"));
      SG_TRY(check_cuda(cudaStreamSynchronize(h->st), "workflow sample"));
      double sip = 0.0, sest = 0.0;
      for (int64_t j = 0; j < want; ++j)
        if (ipv[j] > 0) {
          sip += static_cast<double>(ipv[j]);
          sest += est[j];
        }
      const double cr = sest > 0.0 ? sip / sest : 0.0;
      wf = cr >= 8.0 ? SPGEMM_WORKFLOW_ESTIMATE : SPGEMM_WORKFLOW_SYMBOLIC;
      ws_free(h, d_rows);
      ws_free(h, d_ipv);
      ws_free(h, d_capv);
      ws_free(h, d_est);
    } else {
      wf = SPGEMM_WORKFLOW_SYMBOLIC;  // no light rows to size
    }
  }
  h->workflow = wf;
  h->stats.workflow = wf;
  h->stats.hll_registers = wf == SPGEMM_WORKFLOW_ESTIMATE ? h->hll_m : 0;
  return SPGEMM_OK;
}

// One pass of the light rows into temporary slots: the hash rows listed per ladder level
// (`hrows`, `hstart`), the dense rows from the create bins; every row gets its nnz in `rp` and
// est_nnz, or is marked as overflowed.
void est_pass(spgemm_ctx* h, const int32_t* hrows, const std::vector<int64_t>& hstart, bool dense_rows,
              const EstSink& es, int64_t* rp) {
  Sink sk{};
  sk.row_nnz = rp;
  sk.row_begin = 0;
  sk.row_end = h->m;
  for (int L = 0; L < h->lad.n; ++L) {
    for (int d = 0; d < 2; ++d) {
      if (d == 1 && !dense_rows) continue;
      RowJob job;
      if (d == 0) {
        job.rows = hrows + hstart[L];
        job.count = hstart[L + 1] - hstart[L];
      } else {
        job.rows = h->d_rows + h->bin_start[2 * L + 1];
        job.count = h->bin_start[2 * L + 2] - h->bin_start[2 * L + 1];
      }
      job.slots = h->lad.slots[L];
      job.tpr = h->lad.tpr[L];
      job.dense = d == 1;
      launch_light(h->A, h->B, h->d_span_lo, job, true, sk, h->d_err, h->st, &es);
    }
  }
}

// Light rows under SPGEMM_WORKFLOW_UPPER_BOUND / _ESTIMATE: capacities, one accumulation pass
// into temporary slots (their exact sizes come out of it), and for the rows that did not fit a
// second pass with the IP bound as capacity.  Runs on the handle's stream.
int est_light(spgemm_ctx* h, int64_t* rp) {
  const int nl = h->lad.n;
  const int64_t nlight = h->bin_start[2 * nl];  // light rows: d_rows[0, nlight), bins 0 .. 2nl-1
  if (nlight == 0) return SPGEMM_OK;
  PhaseTimer t(h, 1);
  const bool est = h->workflow == SPGEMM_WORKFLOW_ESTIMATE;
  SG_ALLOC(h->d_est_nnz, int64_t, h->m);
  SG_ALLOC(h->d_row_tmp, int64_t, h->m);
  const int64_t* cap = h->d_ip;
  if (est) {
    SG_TRY(ensure_sketch(h));
    SG_ALLOC(h->d_cap, int64_t, h->m);
    launch_copy_i64(h->d_ip, h->d_cap, h->m, h->st);  // dense rows keep the IP bound
    for (int L = 0; L < nl; ++L)
      launch_hll_rows(h->A, h->d_rows + h->bin_start[2 * L], h->bin_start[2 * L + 1] - h->bin_start[2 * L],
                      h->d_ip, h->d_sketch, h->hll_m, h->hll_coef, h->d_cap, nullptr, h->st);
    cap = h->d_cap;
  }
  // slots in light-row order
  int64_t* off;
  SG_ALLOC(off, int64_t, nlight + 1);
  launch_gather_ip(h->d_rows, nlight, cap, off, h->st);
  SG_TRY(scan(h, off, off, nlight));
  launch_scatter_off(h->d_rows, nlight, off, 0, h->d_row_tmp, h->st);
  int64_t total = 0;
  SG_TRY(check_cuda(cudaMemcpyAsync(&total, off + nlight, sizeof(int64_t), cudaMemcpyDeviceToHost, h->st),
                    "copy slot total"));
  // hash rows of pass 1: the create bins (IP levels), or re-binned by their capacity
  std::vector<int64_t> hstart(nl + 1, 0);
  const int32_t* hrows = h->d_rows;
  int32_t* all = nullptr;
  int32_t* binned = nullptr;
  int64_t nh = 0;
  for (int L = 0; L < nl; ++L) nh += h->bin_start[2 * L + 1] - h->bin_start[2 * L];
  if (est && nh > 0) {
    uint8_t* bin;
    SG_ALLOC(all, int32_t, nh);
    SG_ALLOC(binned, int32_t, nh);
    SG_ALLOC(bin, uint8_t, nh);
    int64_t o = 0;
    for (int L = 0; L < nl; ++L) {
      const int64_t c = h->bin_start[2 * L + 1] - h->bin_start[2 * L];
      if (c) cudaMemcpyAsync(all + o, h->d_rows + h->bin_start[2 * L], sizeof(int32_t) * c, cudaMemcpyDeviceToDevice,
                             h->st);
      o += c;
    }
    launch_val_bins(all, nh, h->d_cap, h->rule, bin, h->st);
    SG_TRY(split_rows(h, all, nh, bin, nl, binned, hstart));
    ws_free(h, bin);
    hrows = binned;
  } else {
    SG_TRY(check_cuda(cudaStreamSynchronize(h->st), "slot total"));
  }
  SG_ALLOC(h->d_tmp_col[0], int32_t, std::max<int64_t>(total, 1));
  SG_ALLOC(h->d_tmp_val[0], double, std::max<int64_t>(total, 1));
  EstSink es{cap, h->d_row_tmp, h->d_tmp_col[0], h->d_tmp_val[0], h->d_est_nnz};
  if (est && nh > 0) {
    est_pass(h, hrows, hstart, true, es, rp);
  } else {  // the create lists: level L's hash rows, then its dense rows
    Sink sk{};
    sk.row_nnz = rp;
    sk.row_begin = 0;
    sk.row_end = h->m;
    for (int L = 0; L < nl; ++L)
      for (int d = 0; d < 2; ++d) {
        RowJob job;
        job.rows = h->d_rows + h->bin_start[2 * L + d];
        job.count = h->bin_start[2 * L + d + 1] - h->bin_start[2 * L + d];
        job.slots = h->lad.slots[L];
        job.tpr = h->lad.tpr[L];
        job.dense = d == 1;
        launch_light(h->A, h->B, h->d_span_lo, job, true, sk, h->d_err, h->st, &es);
      }
  }
  ws_free(h, off);
  // the copy-out lists: rows of the warp bins (short), of the block bins (long), fallback rows
  int wide_level = nl;  // first ladder level served by blocks
  for (int L = nl - 1; L >= 0; --L)
    if (h->lad.tpr[L] > 32) wide_level = L;
  const int64_t split_at = h->bin_start[2 * wide_level];
  h->d_est_list[0] = h->d_rows;
  h->est_count[0] = split_at;
  h->d_est_list[1] = h->d_rows + split_at;
  h->est_count[1] = nlight - split_at;
  h->est_count[2] = 0;
  h->stats.rows_overflow = 0;
  if (!est) return SPGEMM_OK;
  // rows that overflowed their estimated slot: a second pass with the IP bound
  uint8_t* ob;
  int32_t* split;
  std::vector<int64_t> os;
  SG_ALLOC(ob, uint8_t, nlight);
  SG_ALLOC(split, int32_t, nlight);
  launch_overflow_bins(h->d_rows, nlight, h->d_est_nnz, h->d_bin, 2 * wide_level, ob, h->st);
  SG_TRY(split_rows(h, h->d_rows, nlight, ob, 3, split, os));
  ws_free(h, ob);
  const int64_t nover = os[3] - os[2];
  h->d_est_list[0] = split;
  h->est_count[0] = os[1];
  h->d_est_list[1] = split + os[1];
  h->est_count[1] = os[2] - os[1];
  h->stats.rows_overflow = nover;
  if (nover == 0) return SPGEMM_OK;
  const int32_t* over = split + os[2];
  int64_t* off2;
  SG_ALLOC(off2, int64_t, nover + 1);
  launch_gather_ip(over, nover, h->d_ip, off2, h->st);
  SG_TRY(scan(h, off2, off2, nover));
  launch_scatter_off(over, nover, off2, 0, h->d_row_tmp, h->st);
  int64_t total2 = 0;
  SG_TRY(check_cuda(cudaMemcpyAsync(&total2, off2 + nover, sizeof(int64_t), cudaMemcpyDeviceToHost, h->st),
                    "copy fallback total"));
  uint8_t* lb;
  int32_t* obinned;
  std::vector<int64_t> ostart;
  SG_ALLOC(lb, uint8_t, nover);
  SG_ALLOC(obinned, int32_t, nover);
  launch_val_bins(over, nover, h->d_ip, h->rule, lb, h->st);
  SG_TRY(split_rows(h, over, nover, lb, nl, obinned, ostart));  // synchronises: total2 is in
  ws_free(h, lb);
  ws_free(h, off2);
  SG_ALLOC(h->d_tmp_col[1], int32_t, std::max<int64_t>(total2, 1));
  SG_ALLOC(h->d_tmp_val[1], double, std::max<int64_t>(total2, 1));
  EstSink es2{h->d_ip, h->d_row_tmp, h->d_tmp_col[1], h->d_tmp_val[1], h->d_est_nnz};
  est_pass(h, obinned, ostart, false, es2, rp);
  h->d_est_list[2] = obinned;
  h->est_count[2] = nover;
  return SPGEMM_OK;
}

// Enqueue the numeric phase of rows [rb, re) on the handle's stream, written at offset 0 =
// row_ptr[rb] of c_col / c_val; no synchronisation.
int numeric_enqueue(spgemm_ctx* h, int64_t rb, int64_t re, int32_t* c_col, double* c_val) {
  Sink sk{};
  sk.row_ptr = h->c_row_ptr;
  sk.c_col = c_col;
  sk.c_val = c_val;
  sk.row_begin = rb;
  sk.row_end = re;
  if (h->workflow == SPGEMM_WORKFLOW_SYMBOLIC) {
    SG_TRY(numeric_bins(h));
    fork_light(h);
    PhaseTimer t(h, 10, h->st_light);
    light_pass(h, true, sk);
  } else {
    fork_light(h);
    PhaseTimer t(h, 10);
    for (int b = 0; b < 3; ++b)  // light rows: temporary slots -> final positions
      launch_copy_rows(h->d_est_list[b], h->est_count[b], h->d_row_tmp, h->c_row_ptr, rb, re,
                       h->d_tmp_col[b == 2 ? 1 : 0], h->d_tmp_val[b == 2 ? 1 : 0], c_col, c_val, b > 0, h->st);
  }
  if (h->long_rows) SG_TRY(long_pass(h, true, sk));
  bool split = false;
  for (auto& hb : h->batches) {
    if (hb.row_hi < rb || hb.row_lo >= re) continue;
    if (h->fused) {
      if (!split) SG_TRY(fused_prepare(h, true));  // B's current values, split once per call
      split = true;
      SG_TRY(heavy_chunk_numeric(h, hb, sk));
    } else if (!h->resident) {
      SG_TRY(ensure_chat(h, true));
      int64_t* crp;
      SG_ALLOC(crp, int64_t, hb.h1 - hb.h0 + 1);
      if (use_direct(h)) {
        SG_TRY(heavy_direct(h, hb, true, false));
      } else {
        unsigned long long* counts0 = nullptr;
        SG_TRY(alloc_counts0(h, hb, &counts0));
        SG_TRY(heavy_expand(h, hb, true, crp, counts0));
        SG_TRY(heavy_levels(h, hb, true, false, crp, counts0));
        if (counts0) ws_free(h, counts0);
      }
      SG_TRY(heavy_chunk_numeric(h, hb, sk));
      ws_free(h, crp);
    } else {
      SG_TRY(heavy_chunk_numeric(h, hb, sk));
    }
  }
  join_light(h);
  return SPGEMM_OK;
}

void drop_numeric_graph(spgemm_ctx* h) {
  if (h->num_exec) cudaGraphExecDestroy(h->num_exec);
  h->num_exec = nullptr;
  h->num_launches = 0;
}

// Capture the numeric phase of rows [rb, re) into h->num_exec; false (nothing enqueued, the
// stream out of capture) when the capture fails, so the caller runs the phase eagerly.
// The legacy default stream cannot be captured, so the phase is enqueued on a private
// non-blocking stream while the capture is open; the graph is then launched on the caller's.
bool capture_numeric(spgemm_ctx* h, int64_t rb, int64_t re, int32_t* c_col, double* c_val) {
  if (!h->st_graph && cudaStreamCreateWithFlags(&h->st_graph, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    h->st_graph = nullptr;
    return false;
  }
  if (cudaStreamBeginCapture(h->st_graph, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  const long long before = launch_count();
  cudaStream_t caller = h->st;
  h->st = h->st_graph;
  h->capturing = true;
  const int rc = numeric_enqueue(h, rb, re, c_col, c_val);
  h->capturing = false;
  if (rc != SPGEMM_OK) join_light(h);  // keep the light stream joined; the capture is dropped
  h->st = caller;
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(h->st_graph, &g);
  const long long launched = launch_count() - before;
  g_launches.fetch_sub(launched, std::memory_order_relaxed);  // counted again at each replay
  cudaGraphExec_t ex = nullptr;
  const bool ok = rc == SPGEMM_OK && e == cudaSuccess && g &&
                  cudaGraphInstantiate(&ex, g, 0) == cudaSuccess;
  if (g) cudaGraphDestroy(g);
  if (!ok) {
    if (ex) cudaGraphExecDestroy(ex);
    cudaGetLastError();
    // the phase then runs eagerly; the reason stays readable through spgemm_last_error
    set_last_error(std::string("numeric graph capture dropped (ran eagerly): ") +
                   (rc != SPGEMM_OK ? "phase failed under capture" : cudaGetErrorString(e)));
    return false;
  }
  h->num_exec = ex;
  h->num_launches = launched;
  return true;
}

// Numeric phase of rows [rb, re), synchronised.  A repeated call (same rows, same output
// arrays) is captured once into a CUDA graph and replayed from then on, when the phase needs no
// host synchronisation and no allocation: no heavy batch, or the one batch's C^_reord kept from
// the symbolic phase.  Replays cut the launch cost that dominates small products.
int numeric_window(spgemm_ctx* h, int64_t rb, int64_t re, int32_t* c_col, double* c_val) {
  if (h->state < 2) {
    set_last_error("numeric called before symbolic");
    return SPGEMM_ERR_BAD_STATE;
  }
  h->last_graph = false;
  const bool graphable = !h->timing && !(h->opt.flags & SPGEMM_FLAG_NO_GRAPH) && !h->long_rows &&
                         (h->batches.empty() || h->resident || h->fused);
  if (graphable) {
    SG_TRY(numeric_bins(h));  // its one synchronisation stays outside any capture
    const bool same = rb == h->num_rb && re == h->num_re && c_col == h->num_col && c_val == h->num_val;
    if (!same) {
      drop_numeric_graph(h);
      h->num_rb = rb;
      h->num_re = re;
      h->num_col = c_col;
      h->num_val = c_val;
      h->num_calls = 0;
    }
    if (!h->num_exec && h->num_calls >= 1) capture_numeric(h, rb, re, c_col, c_val);
    if (h->num_exec) {
      SG_TRY(check_cuda(cudaGraphLaunch(h->num_exec, h->st), "numeric graph launch"));
      g_launches.fetch_add(h->num_launches, std::memory_order_relaxed);
      h->last_graph = true;
      return sync_and_check(h, "numeric");
    }
    ++h->num_calls;
  }
  SG_TRY(numeric_enqueue(h, rb, re, c_col, c_val));
  return sync_and_check(h, "numeric");
}

// Row windows of the host-streamed numeric phase.  A recomputed heavy batch is expanded once per
// window that intersects its rows, so when batches are not resident every cut falls between two
// batches (each window then holds whole batches); resident products are cut every ~target
// entries of C.
std::vector<int64_t> host_windows(const spgemm_ctx* h, const std::vector<int64_t>& rp, int64_t target) {
  std::vector<int64_t> cuts{0};
  const int64_t m = h->m;
  if ((!h->resident || h->fused) && h->batches.size() > 1) {
    for (size_t b = 1; b < h->batches.size(); ++b) {
      const int64_t c = h->batches[b].row_lo;  // first heavy row of batch b; rows before it belong to earlier windows
      if (c > cuts.back() && rp[c] - rp[cuts.back()] >= target) cuts.push_back(c);
    }
  } else if (h->resident || h->fused || h->batches.empty()) {
    int64_t r = 0;
    while (r < m) {
      // first row whose prefix reaches the next target (binary search on the row pointer)
      const int64_t goal = rp[r] + target;
      int64_t lo = r + 1, hi = m;
      while (lo < hi) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (rp[mid] >= goal) hi = mid; else lo = mid + 1;
      }
      r = lo;
      if (r < m) cuts.push_back(r);
    }
  }
  cuts.push_back(m);
  return cuts;
}

}  // namespace

// ---------------------------------------------------------------------------------------------
extern "C" {

int spgemm_create_ex(spgemm_handle* out, int64_t m, int64_t k, int64_t n, const spgemm_csr* A,
                     const spgemm_csr* B, void* stream, const spgemm_options* opt) {
  g_last_error.clear();
  if (!out) return SPGEMM_ERR_INVALID_ARG;
  *out = nullptr;
  if (m < 0 || k < 0 || n < 0 || !valid_csr_desc(A, m, k) || !valid_csr_desc(B, k, n)) {
    set_last_error("invalid shapes or CSR descriptors");
    return SPGEMM_ERR_INVALID_ARG;
  }
  if (n > 0x7fffffffLL || k > 0x7fffffffLL || m > 0x7fffffffLL) {
    set_last_error("dimensions beyond int32 indices");
    return SPGEMM_ERR_OVERFLOW;
  }
  spgemm_ctx* h = new spgemm_ctx();
  h->m = m;
  h->k = k;
  h->n = n;
  h->A = *A;
  h->B = *B;
  h->st = static_cast<cudaStream_t>(stream);
  if (opt) h->opt = *opt;
  if (h->opt.workflow < SPGEMM_WORKFLOW_SYMBOLIC || h->opt.workflow > SPGEMM_WORKFLOW_AUTO ||
      (h->opt.hll_registers != 0 && !hll_registers_ok(h->opt.hll_registers)) || !(h->opt.hll_coef >= 0.0)) {
    delete h;
    set_last_error("invalid workflow, register count or coefficient");
    return SPGEMM_ERR_INVALID_ARG;
  }
  const char* tenv = getenv("SPGEMM_TIMING");
  h->timing = (tenv && tenv[0] == '1') || (h->opt.flags & SPGEMM_FLAG_TIMING);
  int rc = SPGEMM_OK;
  auto fail = [&](int code) {
    spgemm_destroy(h);
    return code;
  };
  int dev = 0, sms = 0, optin = 0, l2 = 0;
  if ((rc = check_cuda(cudaGetDevice(&dev), "cudaGetDevice")) != SPGEMM_OK) return fail(rc);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
  h->device = dev;
  h->pool = device_pool(dev);
  if (!h->pool) {
    set_last_error("could not create the device memory pool");
    return fail(SPGEMM_ERR_CUDA);
  }
  h->sms = sms;
  h->smem_optin = optin;
  h->l2_bytes = l2;
  const int64_t s_lm = h->opt.smem_bytes ? h->opt.smem_bytes : optin - kSmemReserve;
  if (s_lm + kSmemReserve > optin) {
    set_last_error("smem_bytes exceeds the device's shared memory per block");
    return fail(SPGEMM_ERR_INVALID_ARG);
  }
  // The dense chunk accumulator runs kDenseBlocksPerSm blocks per SM (their per-chunk phases
  // overlap; one 16,384-wide block per SM measured 22.4 ms against 18.1 ms for three 8,192-wide
  // ones on R-MAT scale 18), so unless the caller fixes W its local memory is that share of the
  // SM's shared memory: W is the widest power of two whose dense block (values, bitmap, word
  // prefix, hub copies) fits in the share, the dense width of Eq. 5 for that s_LM.
  spgemm_options popt = h->opt;
  if (!popt.chunk_width && !popt.smem_bytes) {
    int smem_sm = 0;
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    const size_t share = static_cast<size_t>(smem_sm / kDenseBlocksPerSm) - 1024;  // 1 KB per block for the system
    int64_t w = 0;
    for (int64_t c = 1024; c <= (int64_t(1) << 24) && chunk_smem_bytes(c, 0, 2, false) <= share; c *= 2) w = c;
    if (w) popt.chunk_width = w;
  }
  if ((rc = plan_params(n, s_lm, &popt, &h->plan)) != SPGEMM_OK) {
    set_last_error("planner rejected the options");
    return fail(rc);
  }
  h->lad = make_ladder(h->plan.tau);
  if (h->opt.debug_hash_slots > 0)  // tests: tables too small for the longer rows
    for (int i = 0; i < h->lad.n; ++i) h->lad.slots[i] = std::min<int64_t>(h->lad.slots[i], h->opt.debug_hash_slots);
  // the largest light bin's hash table must fit one block's shared memory (this also keeps the
  // products of a light row, at most tau, far below 2^31)
  if (light_smem_bytes(h->lad.slots[h->lad.n - 1], h->lad.tpr[h->lad.n - 1], false, true) > static_cast<size_t>(optin)) {
    set_last_error("tau too large: the light-row hash table does not fit in shared memory");
    return fail(SPGEMM_ERR_INVALID_ARG);
  }
  h->rule.n = h->lad.n;
  for (int i = 0; i < h->lad.n; ++i) {
    h->rule.upper[i] = h->lad.upper[i];
    h->rule.slots[i] = h->lad.slots[i];
  }
  h->rule.tau = h->plan.tau;
  h->rule.all_heavy = (h->opt.flags & SPGEMM_FLAG_ALL_HEAVY) ? 1 : 0;
  h->rule.all_light = (h->opt.flags & SPGEMM_FLAG_ALL_LIGHT) ? 1 : 0;
  h->rule.no_dense = (h->opt.flags & SPGEMM_FLAG_NO_DENSE_LIGHT) ? 1 : 0;
  h->nbins = 2 * h->lad.n + 1;
  if (!(h->opt.flags & SPGEMM_FLAG_NO_ESC))
    while (h->esc_levels < h->lad.n && h->lad.upper[h->esc_levels] <= esc_max_products()) ++h->esc_levels;

  PhaseTimer* tsetup = new PhaseTimer(h, 0);
  h->d_err = static_cast<uint32_t*>(ws_alloc(h, sizeof(uint32_t)));
  if (!h->d_err) {
    delete tsetup;
    return fail(SPGEMM_ERR_OUT_OF_MEMORY);
  }
  cudaMemsetAsync(h->d_err, 0, sizeof(uint32_t), h->st);
  h->st_light = pooled_stream(dev);
  h->ev_fork = pooled_event(dev);
  h->ev_join = pooled_event(dev);
  if (!h->st_light || !h->ev_fork || !h->ev_join) {
    delete tsetup;
    set_last_error("stream or event creation failed");
    return fail(SPGEMM_ERR_CUDA);
  }
  h->d_counter = static_cast<int*>(ws_alloc(h, sizeof(int)));
  if (!h->d_counter) {
    delete tsetup;
    return fail(SPGEMM_ERR_OUT_OF_MEMORY);
  }
  auto body = [&]() -> int {
    if (h->opt.flags & SPGEMM_FLAG_VALIDATE) {
      launch_validate(h->A, h->d_err, h->st);
      launch_validate(h->B, h->d_err, h->st);
      SG_TRY(sync_and_check(h, "input validation"));
    }
    const int64_t mm = std::max<int64_t>(m, 1);
    SG_ALLOC(h->d_ip, int64_t, mm);
    SG_ALLOC(h->d_span_lo, int32_t, mm);
    SG_ALLOC(h->d_bin, uint8_t, mm);
    SG_ALLOC(h->d_rows, int32_t, mm);
    int32_t *bmin, *bmax;
    SG_ALLOC(bmin, int32_t, std::max<int64_t>(k, 1));
    SG_ALLOC(bmax, int32_t, std::max<int64_t>(k, 1));
    launch_brow_minmax(h->B, bmin, bmax, h->st);
    launch_row_ip(h->A, h->B, bmin, bmax, h->rule, h->d_ip, h->d_span_lo, h->d_bin, h->st);
    const int nb = h->nbins;
    const int64_t nblk = bin_blocks(m);
    int64_t* starts;
    SG_ALLOC(h->d_binoff, int64_t, nb * nblk + 1);
    SG_ALLOC(starts, int64_t, nb + 1);
    cudaMemsetAsync(h->d_binoff, 0, sizeof(int64_t) * (nb * nblk + 1), h->st);
    launch_bin_count(h->d_bin, m, nb, h->d_binoff, h->st);
    SG_TRY(scan(h, h->d_binoff, h->d_binoff, nb * nblk));
    launch_bin_scatter(h->d_bin, m, nb, h->d_binoff, h->d_rows, h->st);
    launch_bin_starts(h->d_binoff, nblk, nb, starts, h->st);
    h->bin_start.assign(nb + 1, 0);
    SG_TRY(check_cuda(cudaMemcpyAsync(h->bin_start.data(), starts, sizeof(int64_t) * (nb + 1),
                                      cudaMemcpyDeviceToHost, h->st), "copy bin starts"));
    SG_TRY(sync_and_check(h, "setup"));
    ws_free(h, bmin);
    ws_free(h, bmax);
    ws_free(h, starts);
    // heavy rows and their IP prefix
    const int hb = 2 * h->lad.n;
    h->nheavy = h->bin_start[hb + 1] - h->bin_start[hb];
    h->d_heavy = h->d_rows + h->bin_start[hb];
    // statistics
    std::vector<int64_t> hip(1, 0);
    h->stats.m = m;
    h->stats.k = k;
    h->stats.n = n;
    h->stats.c_nnz = -1;
    h->stats.rows_heavy = h->nheavy;
    h->stats.rows_light = h->bin_start[hb] - h->bin_start[0];
    h->stats.rows_empty = m - h->bin_start[nb];
    for (int L = 0; L < h->lad.n; ++L)
      h->stats.rows_dense_light += h->bin_start[2 * L + 2] - h->bin_start[2 * L + 1];
    {
      // total IP (for the statistics): scan of IP per row
      int64_t* tmp;
      SG_ALLOC(tmp, int64_t, m + 1);
      SG_TRY(scan(h, h->d_ip, tmp, m));
      SG_TRY(check_cuda(cudaMemcpyAsync(&h->stats.ip_total, tmp + m, sizeof(int64_t), cudaMemcpyDeviceToHost,
                                        h->st), "copy ip total"));
      SG_TRY(check_cuda(cudaStreamSynchronize(h->st), "ip total"));
      ws_free(h, tmp);
    }
    if (h->nheavy > 0 && (h->opt.flags & SPGEMM_FLAG_LONG_ROWS) && h->n <= 0x7fffffffLL) {
      // heavy rows by the long-row hash: no expansion, no batches
      h->long_rows = true;
      h->stats.long_rows = 1;
      std::vector<int64_t> hp(h->nheavy + 1);
      SG_ALLOC(h->d_heavy_pre, int64_t, h->nheavy + 1);
      launch_gather_ip(h->d_heavy, h->nheavy, h->d_ip, h->d_heavy_pre, h->st);
      SG_TRY(scan(h, h->d_heavy_pre, h->d_heavy_pre, h->nheavy));
      SG_TRY(check_cuda(cudaMemcpyAsync(hp.data(), h->d_heavy_pre + h->nheavy, sizeof(int64_t), cudaMemcpyDeviceToHost,
                                        h->st), "copy heavy IP"));
      SG_TRY(check_cuda(cudaStreamSynchronize(h->st), "heavy IP"));
      h->stats.ip_heavy = hp[0];
    } else if (h->nheavy > 0) {
      h->fused = (h->opt.flags & SPGEMM_FLAG_FUSED) && h->plan.chunks_required <= kFusedMaxChunks &&
                 h->B.nnz < (int64_t(1) << 31);
      h->stats.fused = h->fused ? 1 : 0;
      SG_ALLOC(h->d_heavy_pre, int64_t, h->nheavy + 1);
      launch_gather_ip(h->d_heavy, h->nheavy, h->d_ip, h->d_heavy_pre, h->st);
      SG_TRY(scan(h, h->d_heavy_pre, h->d_heavy_pre, h->nheavy));
      h->heavy_pre.resize(h->nheavy + 1);
      std::vector<int32_t> hrows(h->nheavy);
      SG_TRY(check_cuda(cudaMemcpyAsync(h->heavy_pre.data(), h->d_heavy_pre, sizeof(int64_t) * (h->nheavy + 1),
                                        cudaMemcpyDeviceToHost, h->st), "copy heavy prefix"));
      SG_TRY(check_cuda(cudaMemcpyAsync(hrows.data(), h->d_heavy, sizeof(int32_t) * h->nheavy,
                                        cudaMemcpyDeviceToHost, h->st), "copy heavy rows"));
      SG_TRY(check_cuda(cudaStreamSynchronize(h->st), "heavy prefix"));
      h->stats.ip_heavy = h->heavy_pre[h->nheavy];
      // batches of heavy rows whose C^ fits the budget
      int64_t cap = h->opt.heavy_batch_elems;
      if (!cap) {
        // free device memory plus what the handle's pool holds cached but unused (a previous
        // product's workspace, reused by this one's allocations)
        size_t fr = 0, tot = 0;
        cudaMemGetInfo(&fr, &tot);
        uint64_t reserved = 0, used = 0;
        if (cudaMemPoolGetAttribute(h->pool, cudaMemPoolAttrReservedMemCurrent, &reserved) != cudaSuccess ||
            cudaMemPoolGetAttribute(h->pool, cudaMemPoolAttrUsedMemCurrent, &used) != cudaSuccess) {
          cudaGetLastError();
          reserved = used = 0;
        }
        const double avail = static_cast<double>(fr) + static_cast<double>(reserved > used ? reserved - used : 0);
        // 24 bytes per element: column + value, twice for the multisplit's double buffer.  The
        // direct split allocates one half only and keeps the same batches: twice their size
        // measured no faster (R-MAT scale 21: 27 batches 3.20 s against 49 batches 3.18-3.22 s
        // per product), and the smaller ones leave the memory to the caller's C
        cap = static_cast<int64_t>(avail * 0.35 / 24.0);
      }
      int64_t i = 0, maxb = 0;
      while (i < h->nheavy) {
        HeavyBatch b;
        b.h0 = i;
        int64_t j = i + 1;
        while (j < h->nheavy && h->heavy_pre[j + 1] - h->heavy_pre[i] <= cap) ++j;
        b.h1 = j;
        b.elems = h->heavy_pre[j] - h->heavy_pre[i];
        b.row_lo = hrows[i];
        b.row_hi = hrows[j - 1];
        maxb = std::max(maxb, b.elems);
        h->batches.push_back(b);
        i = j;
      }
      h->batch_cap = (maxb + 15) / 16 * 16;  // keeps both halves of the C^ buffer 16-byte aligned
      h->resident = h->batches.size() == 1 && !(h->opt.flags & SPGEMM_FLAG_RECOMPUTE) && !h->fused;
      // a recomputed expansion need not run in the symbolic phase: its chunks are counted from
      // generated products (the column split of B), the numeric phase expands once, with values
      h->gen_symbolic = !h->fused && !h->resident && use_direct(h) && !(h->opt.flags & SPGEMM_FLAG_NO_GEN_SYMBOLIC) &&
                        h->plan.chunks_required <= kFusedMaxChunks && h->B.nnz < (int64_t(1) << 31);
      h->stats.gen_symbolic = h->gen_symbolic ? 1 : 0;
      h->stats.heavy_batches = static_cast<int64_t>(h->batches.size());
      h->stats.chat_bytes = h->fused ? 0 : maxb * 12;
      h->stats.resident = h->resident ? 1 : 0;
    }
    return SPGEMM_OK;
  };
  rc = body();
  delete tsetup;
  if (rc != SPGEMM_OK) return fail(rc);
  h->state = 1;
  *out = h;
  return SPGEMM_OK;
}

int spgemm_create(spgemm_handle* h, int64_t m, int64_t k, int64_t n, const spgemm_csr* A, const spgemm_csr* B,
                  void* stream) {
  return spgemm_create_ex(h, m, k, n, A, B, stream, nullptr);
}

int spgemm_symbolic(spgemm_handle h, int64_t* c_row_ptr, int64_t* c_nnz) {
  g_last_error.clear();
  if (!h || !c_row_ptr || !c_nnz) return SPGEMM_ERR_INVALID_ARG;
  if (h->state != 1) {
    set_last_error("symbolic must follow create, once");
    return SPGEMM_ERR_BAD_STATE;
  }
  cudaMemsetAsync(c_row_ptr, 0, sizeof(int64_t) * (h->m + 1), h->st);
  Sink sk{};
  sk.row_nnz = c_row_ptr;
  sk.row_begin = 0;
  sk.row_end = h->m;
  SG_TRY(choose_workflow(h));
  if (h->workflow != SPGEMM_WORKFLOW_SYMBOLIC) SG_TRY(est_light(h, c_row_ptr));
  fork_light(h);
  if (h->workflow == SPGEMM_WORKFLOW_SYMBOLIC) {
    PhaseTimer t(h, 1, h->st_light);
    light_pass(h, false, sk);
  }
  int64_t levels = 0, finals = 0, dense = 0;
  if (h->long_rows) SG_TRY(long_pass(h, false, sk));
  if ((h->fused || h->gen_symbolic) && !h->batches.empty()) SG_TRY(fused_prepare(h, false));
  for (auto& hb : h->batches) {
    if (h->fused || h->gen_symbolic) {
      SG_TRY(heavy_fused(h, hb));
      SG_TRY(heavy_chunk_symbolic(h, hb, c_row_ptr));
      levels = std::max<int64_t>(levels, 1);
      finals += hb.nfinal;
      dense += hb.f_bin_start[h->lad.n + 4] - hb.f_bin_start[h->lad.n + 3];
      continue;
    }
    const bool vals = h->resident;
    SG_TRY(ensure_chat(h, vals));
    int64_t* crp;
    SG_ALLOC(crp, int64_t, hb.h1 - hb.h0 + 1);
    if (use_direct(h)) {
      SG_TRY(heavy_direct(h, hb, vals, true));
    } else {
      unsigned long long* counts0 = nullptr;
      SG_TRY(alloc_counts0(h, hb, &counts0));
      SG_TRY(heavy_expand(h, hb, vals, crp, counts0));
      SG_TRY(heavy_levels(h, hb, vals, true, crp, counts0));
      if (counts0) ws_free(h, counts0);
    }
    SG_TRY(heavy_chunk_symbolic(h, hb, c_row_ptr));
    ws_free(h, crp);
    levels = std::max<int64_t>(levels, static_cast<int64_t>(hb.lv.size()));
    finals += hb.nfinal;
    dense += hb.f_bin_start[h->lad.n + 4] - hb.f_bin_start[h->lad.n + 3];
  }
  join_light(h);
  h->stats.levels_run = levels;
  h->stats.direct_split = (!h->fused && !h->batches.empty() && use_direct(h)) ? 1 : 0;
  h->stats.final_chunks = finals;
  h->stats.chunks_dense = dense;
  {
    PhaseTimer t(h, 9);
    SG_TRY(scan(h, c_row_ptr, c_row_ptr, h->m));
  }
  // nnz(C) and the numeric bins of the light rows come back with the one synchronisation
  int64_t nnz = 0;
  HostStatus* hs = host_status();
  bool bins_pending = false;
  if (hs) {
    h->nbin_start.clear();
    if (h->workflow == SPGEMM_WORKFLOW_SYMBOLIC) SG_TRY(numeric_bins_enqueue(h, c_row_ptr, hs->starts));
    bins_pending = h->nbin_start.empty() && h->workflow == SPGEMM_WORKFLOW_SYMBOLIC;
    SG_TRY(check_cuda(cudaMemcpyAsync(&hs->nnz, c_row_ptr + h->m, sizeof(int64_t), cudaMemcpyDeviceToHost, h->st),
                      "copy nnz"));
    SG_TRY(sync_and_check(h, "symbolic"));
    nnz = hs->nnz;
    if (bins_pending) h->nbin_start.assign(hs->starts, hs->starts + h->lad.n + 1);
  } else {
    SG_TRY(check_cuda(cudaMemcpyAsync(&nnz, c_row_ptr + h->m, sizeof(int64_t), cudaMemcpyDeviceToHost, h->st),
                      "copy nnz"));
    SG_TRY(sync_and_check(h, "symbolic"));
  }
  *c_nnz = nnz;
  h->stats.c_nnz = nnz;
  h->stats.c_nnz_heavy = 0;
  h->stats.dense_elems = 0;
  h->stats.dense_nnz = 0;
  for (auto& hb : h->batches) {
    h->stats.c_nnz_heavy += hb.nnz_c;
    h->stats.dense_elems += hb.dense_sums[0];
    h->stats.dense_nnz += hb.dense_sums[1];
  }
  h->c_row_ptr = c_row_ptr;
  h->state = 2;
  return SPGEMM_OK;
}

int spgemm_numeric(spgemm_handle h, int32_t* c_col_idx, double* c_vals) {
  g_last_error.clear();
  if (!h) return SPGEMM_ERR_INVALID_ARG;
  if (h->stats.c_nnz > 0 && (!c_col_idx || !c_vals)) return SPGEMM_ERR_INVALID_ARG;
  return numeric_window(h, 0, h->m, c_col_idx, c_vals);
}

int spgemm_numeric_rows(spgemm_handle h, int64_t row_begin, int64_t row_end, int32_t* c_col_idx,
                        double* c_vals) {
  g_last_error.clear();
  if (!h) return SPGEMM_ERR_INVALID_ARG;
  if (row_begin < 0 || row_end > h->m || row_begin > row_end) {
    set_last_error("row range outside [0, m]");
    return SPGEMM_ERR_INVALID_ARG;
  }
  if (row_begin == row_end) return SPGEMM_OK;
  if (!c_col_idx || !c_vals) return SPGEMM_ERR_INVALID_ARG;
  return numeric_window(h, row_begin, row_end, c_col_idx, c_vals);
}

int spgemm_numeric_host(spgemm_handle h, int64_t* c_row_ptr, int32_t* c_col_idx, double* c_vals,
                        int64_t window_nnz) {
  g_last_error.clear();
  if (!h || window_nnz < 0) return SPGEMM_ERR_INVALID_ARG;
  if (h->state < 2) {
    set_last_error("numeric called before symbolic");
    return SPGEMM_ERR_BAD_STATE;
  }
  const int64_t nnz = h->stats.c_nnz, m = h->m;
  if (nnz > 0 && (!c_col_idx || !c_vals)) return SPGEMM_ERR_INVALID_ARG;
  std::vector<int64_t> rp(static_cast<size_t>(m + 1));
  SG_TRY(check_cuda(cudaMemcpyAsync(rp.data(), h->c_row_ptr, sizeof(int64_t) * (m + 1), cudaMemcpyDeviceToHost, h->st),
                    "copy row_ptr"));
  SG_TRY(check_cuda(cudaStreamSynchronize(h->st), "copy row_ptr"));
  if (c_row_ptr) std::copy(rp.begin(), rp.end(), c_row_ptr);
  if (nnz == 0) return spgemm_numeric(h, nullptr, nullptr);
  // default window: a quarter of C, at least 4 M entries, staging at most a fifth of free memory
  size_t free_b = 0, total_b = 0;
  cudaMemGetInfo(&free_b, &total_b);
  int64_t target = window_nnz ? window_nnz : std::max<int64_t>(nnz / 4, int64_t(1) << 22);
  target = std::min<int64_t>(target, std::max<int64_t>(1, static_cast<int64_t>(free_b / 5 / 24)));
  const std::vector<int64_t> cuts = host_windows(h, rp, target);
  int64_t wmax = 0;
  for (size_t w = 0; w + 1 < cuts.size(); ++w) wmax = std::max(wmax, rp[cuts[w + 1]] - rp[cuts[w]]);
  if (!h->st_copy && cudaStreamCreateWithFlags(&h->st_copy, cudaStreamNonBlocking) != cudaSuccess) {
    set_last_error("copy stream creation failed");
    return SPGEMM_ERR_CUDA;
  }
  for (int b = 0; b < 2; ++b) {
    if (!h->ev_done[b] && cudaEventCreateWithFlags(&h->ev_done[b], cudaEventDisableTiming) != cudaSuccess)
      return SPGEMM_ERR_CUDA;
    if (!h->ev_copied[b] && cudaEventCreateWithFlags(&h->ev_copied[b], cudaEventDisableTiming) != cudaSuccess)
      return SPGEMM_ERR_CUDA;
  }
  // two staging buffers: window w is computed into buffer w % 2 while window w - 1 is copied out
  const int nbuf = cuts.size() > 2 ? 2 : 1;
  int32_t* scol[2] = {nullptr, nullptr};
  double* sval[2] = {nullptr, nullptr};
  for (int b = 0; b < nbuf; ++b) {
    SG_ALLOC(scol[b], int32_t, wmax);
    SG_ALLOC(sval[b], double, wmax);
  }
  int rc = SPGEMM_OK;
  for (size_t w = 0; w + 1 < cuts.size() && rc == SPGEMM_OK; ++w) {
    const int b = static_cast<int>(w % nbuf);
    const int64_t rb = cuts[w], re = cuts[w + 1], off = rp[rb], cnt = rp[re] - rp[rb];
    if (w >= static_cast<size_t>(nbuf)) cudaStreamWaitEvent(h->st, h->ev_copied[b], 0);  // buffer free again
    rc = numeric_enqueue(h, rb, re, scol[b], sval[b]);
    if (rc != SPGEMM_OK) break;
    cudaEventRecord(h->ev_done[b], h->st);
    cudaStreamWaitEvent(h->st_copy, h->ev_done[b], 0);
    if (cnt > 0) {
      cudaMemcpyAsync(c_col_idx + off, scol[b], sizeof(int32_t) * cnt, cudaMemcpyDeviceToHost, h->st_copy);
      cudaMemcpyAsync(c_vals + off, sval[b], sizeof(double) * cnt, cudaMemcpyDeviceToHost, h->st_copy);
    }
    cudaEventRecord(h->ev_copied[b], h->st_copy);
  }
  // the handle's stream waits for the last copies, so the staging buffers are freed after them
  for (int b = 0; b < nbuf; ++b) cudaStreamWaitEvent(h->st, h->ev_copied[b], 0);
  for (int b = 0; b < nbuf; ++b) {
    ws_free(h, scol[b]);
    ws_free(h, sval[b]);
  }
  if (rc != SPGEMM_OK) {
    cudaStreamSynchronize(h->st_copy);
    cudaStreamSynchronize(h->st);
    return rc;
  }
  SG_TRY(check_cuda(cudaStreamSynchronize(h->st_copy), "numeric host copies"));
  return sync_and_check(h, "numeric");
}

int spgemm_row_windows(spgemm_handle h, int64_t target_nnz, int64_t* cuts, int64_t cap, int64_t* n_windows,
                       int64_t* max_window_nnz) {
  g_last_error.clear();
  if (!h || target_nnz < 0 || cap < 0 || !n_windows || (cap > 0 && !cuts)) return SPGEMM_ERR_INVALID_ARG;
  if (h->state < 2) {
    set_last_error("row windows need the symbolic phase");
    return SPGEMM_ERR_BAD_STATE;
  }
  const int64_t m = h->m;
  std::vector<int64_t> rp(static_cast<size_t>(m + 1));
  SG_TRY(check_cuda(cudaMemcpyAsync(rp.data(), h->c_row_ptr, sizeof(int64_t) * (m + 1), cudaMemcpyDeviceToHost, h->st),
                    "copy row_ptr"));
  SG_TRY(check_cuda(cudaStreamSynchronize(h->st), "copy row_ptr"));
  const int64_t target = target_nnz ? target_nnz : std::max<int64_t>(rp[m] / 4, int64_t(1) << 22);
  const std::vector<int64_t> c = host_windows(h, rp, target);
  const int64_t nw = static_cast<int64_t>(c.size()) - 1;
  *n_windows = nw;
  int64_t wmax = 0;
  for (int64_t w = 0; w < nw; ++w) wmax = std::max(wmax, rp[c[w + 1]] - rp[c[w]]);
  if (max_window_nnz) *max_window_nnz = wmax;
  if (cap < nw + 1) {
    set_last_error("cuts array too short: it needs n_windows + 1 entries");
    return SPGEMM_ERR_INVALID_ARG;
  }
  std::copy(c.begin(), c.end(), cuts);
  return SPGEMM_OK;
}

int spgemm_get_stats(spgemm_handle h, spgemm_stats* out) {
  if (!h || !out) return SPGEMM_ERR_INVALID_ARG;
  *out = h->stats;
  out->numeric_graph = h->last_graph ? 1 : 0;
  return SPGEMM_OK;
}

int spgemm_get_plan(spgemm_handle h, spgemm_plan* out) {
  if (!h || !out) return SPGEMM_ERR_INVALID_ARG;
  *out = h->plan;
  return SPGEMM_OK;
}

int spgemm_get_phase_times(spgemm_handle h, double* t, int64_t* launches, int32_t count) {
  if (!h || !t || count < 0) return SPGEMM_ERR_INVALID_ARG;
  drain_timers(h);
  for (int i = 0; i < count && i < kPhaseSlots; ++i) {
    t[i] = h->phase_ms[i];
    if (launches) launches[i] = h->phase_n[i];
  }
  return SPGEMM_OK;
}

long long spgemm_kernel_launches(void) { return launch_count(); }

namespace {
bool csr_ok(const spgemm_csr* C) {
  return C && C->rows >= 0 && C->cols >= 0 && C->nnz >= 0 && C->row_ptr && (C->nnz == 0 || (C->col_idx && C->vals));
}
}  // namespace

int spgemm_mcl_prune_symbolic(const spgemm_csr* C, double threshold, double* col_sums, int64_t* out_row_ptr,
                              int64_t* out_nnz, void* stream) {
  g_last_error.clear();
  if (!csr_ok(C) || !out_row_ptr || !out_nnz || (C->cols > 0 && !col_sums) || !(threshold >= 0.0))
    return SPGEMM_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (C->cols > 0) cudaMemsetAsync(col_sums, 0, sizeof(double) * C->cols, st);
  launch_col_sums(*C, col_sums, st);
  cudaMemsetAsync(out_row_ptr, 0, sizeof(int64_t) * (C->rows + 1), st);
  launch_keep_count(*C, col_sums, threshold, out_row_ptr, st);
  int64_t* scratch = nullptr;
  const int64_t need = std::max<int64_t>(scan_scratch_elems(C->rows), 1);
  if (cudaMallocAsync(reinterpret_cast<void**>(&scratch), sizeof(int64_t) * need, st) != cudaSuccess) {
    cudaGetLastError();
    set_last_error("scan scratch allocation failed");
    return SPGEMM_ERR_OUT_OF_MEMORY;
  }
  scan_excl_i64(out_row_ptr, out_row_ptr, C->rows, scratch, st);
  cudaFreeAsync(scratch, st);
  int64_t nnz = 0;
  SG_TRY(check_cuda(cudaMemcpyAsync(&nnz, out_row_ptr + C->rows, sizeof(int64_t), cudaMemcpyDeviceToHost, st),
                    "copy pruned nnz"));
  SG_TRY(check_cuda(cudaStreamSynchronize(st), "mcl prune symbolic"));
  *out_nnz = nnz;
  return SPGEMM_OK;
}

int spgemm_mcl_prune_numeric(const spgemm_csr* C, double threshold, const double* col_sums,
                             const int64_t* out_row_ptr, int32_t* out_col, double* out_val, void* stream) {
  g_last_error.clear();
  if (!csr_ok(C) || !out_row_ptr || (C->nnz > 0 && (!col_sums || !out_col || !out_val)) || !(threshold >= 0.0))
    return SPGEMM_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  launch_keep_write(*C, col_sums, threshold, out_row_ptr, out_col, out_val, st);
  return check_cuda(cudaGetLastError(), "mcl prune numeric");
}

int spgemm_hll_estimate(const spgemm_csr* A, const spgemm_csr* B, int32_t registers, double coef, int64_t* cap,
                        void* stream) {
  g_last_error.clear();
  if (!A || !B || !cap || A->rows < 0 || B->rows < 0 || A->cols != B->rows || !hll_registers_ok(registers) ||
      !(coef > 0.0))
    return SPGEMM_ERR_INVALID_ARG;
  if (A->rows == 0) return SPGEMM_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* sk = nullptr;
  int64_t* ip = nullptr;
  if (cudaMallocAsync(reinterpret_cast<void**>(&sk), std::max<int64_t>(B->rows, 1) * registers, st) != cudaSuccess ||
      cudaMallocAsync(reinterpret_cast<void**>(&ip), sizeof(int64_t) * A->rows, st) != cudaSuccess) {
    cudaGetLastError();
    if (sk) cudaFreeAsync(sk, st);
    set_last_error("sketch allocation failed");
    return SPGEMM_ERR_OUT_OF_MEMORY;
  }
  launch_hll_sketch(*B, registers, sk, st);
  launch_row_products(*A, *B, ip, st);
  launch_hll_rows(*A, nullptr, A->rows, ip, sk, registers, coef, cap, nullptr, st);
  cudaFreeAsync(sk, st);
  cudaFreeAsync(ip, st);
  return check_cuda(cudaGetLastError(), "hll estimate");
}

int spgemm_destroy(spgemm_handle h) {
  if (!h) return SPGEMM_OK;
  drain_timers(h);
  if (h->st_light) cudaStreamSynchronize(h->st_light);
  drop_numeric_graph(h);
  if (h->st_graph) cudaStreamDestroy(h->st_graph);
  for (void* p : h->allocs) cudaFreeAsync(p, h->st);
  h->allocs.clear();
  h->alloc_bytes.clear();
  h->ws_bytes = 0;
  cudaStreamSynchronize(h->st);
  for (int b = 0; b < 2; ++b) {
    if (h->ev_done[b]) cudaEventDestroy(h->ev_done[b]);
    if (h->ev_copied[b]) cudaEventDestroy(h->ev_copied[b]);
  }
  if (h->st_copy) cudaStreamDestroy(h->st_copy);
  return_event(h->device, h->ev_fork);
  return_event(h->device, h->ev_join);
  return_stream(h->device, h->st_light);  // synchronised above
  delete h;
  return SPGEMM_OK;
}

int spgemm_release_memory(void) {
  {
    std::lock_guard<std::mutex> lock(g_pool_mu);
    for (int d = 0; d < 64; ++d)
      if (g_pool[d]) cudaMemPoolTrimTo(g_pool[d], 0);
  }
  std::lock_guard<std::mutex> lock(g_sp_mu);
  for (int d = 0; d < 64; ++d) {
    for (cudaStream_t st : g_sp_streams[d]) cudaStreamDestroy(st);
    for (cudaEvent_t e : g_sp_events[d]) cudaEventDestroy(e);
    g_sp_streams[d].clear();
    g_sp_events[d].clear();
  }
  return SPGEMM_OK;
}

const char* spgemm_strerror(int code) {
  switch (code) {
    case SPGEMM_OK: return "ok";
    case SPGEMM_ERR_INVALID_ARG: return "invalid argument";
    case SPGEMM_ERR_INVALID_CSR: return "malformed CSR input";
    case SPGEMM_ERR_BAD_STATE: return "call out of order";
    case SPGEMM_ERR_OUT_OF_MEMORY: return "out of device memory";
    case SPGEMM_ERR_OVERFLOW: return "size exceeds the index types";
    case SPGEMM_ERR_DEVICE: return "device-side check failed";
    case SPGEMM_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

const char* spgemm_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
