// Internal declarations of the SpGEMM library: handle, plan constants, kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/spgemm.h"
#include "common.cuh"

namespace sg {

// ---- tile sizes shared by the planner and the kernels ---------------------------------
constexpr int64_t kMsTile = 1024;          // elements per histogram / multisplit tile
constexpr int kMsThreads = 128;            // threads per multisplit block (8 elements each)
constexpr int64_t kMsSmemBudget = 65536;   // bytes of shared memory per multisplit block (Eq. 6)
constexpr int64_t kMsMaxBins = 2048;       // group_rows * chunks bins held by one block
constexpr int64_t kOpTile = 1024;          // elements per outer-product block
constexpr int kOpThreads = 128;            // (small blocks: 2048/256 measured 0.4 ms slower on R-MAT s18)
constexpr int64_t kOdTile = 4096;          // products per block of the direct split
constexpr int kOdWin = 256;                // entries of a direct-split tile staged at a time
constexpr int kSmemReserve = 7168;         // bytes kept back from s_LM for per-block staging
constexpr int kMaxLadder = 16;             // light bin ladder levels
constexpr int kScanTile = 4096;            // elements per scan block (512 threads x 8)
constexpr int kPhaseSlots = 13;            // timed regions, see spgemm_get_phase_times
constexpr int64_t kChunkDenseMin = 1024;   // last-level chunks above this size use the dense accumulator
constexpr int kDenseBlocksPerSm = 3;        // dense chunk accumulator blocks per SM (sets the default W)

// Light-row / chunk bin ladder derived from tau (hash tables at load factor 1/2).
struct Ladder {
  int n = 0;                       // levels
  int64_t upper[kMaxLadder];       // level L takes IP (or chunk size) in (upper[L-1], upper[L]]
  int64_t slots[kMaxLadder];       // hash slots = 2 * upper (shortened dense: span <= slots)
  int tpr[kMaxLadder];             // threads per row: 32 = one warp per row, else one block
};

// Parameters of the row classifier, passed by value to kernels.
struct BinRule {
  int n;                 // ladder levels
  int64_t upper[kMaxLadder];
  int64_t slots[kMaxLadder];
  int64_t tau;
  int all_heavy, all_light, no_dense;
};

// Bin numbering: level L hash = 2L, level L dense = 2L+1, heavy = 2n, empty = 255.
constexpr uint8_t kBinEmpty = 255;

// ---- launch accounting --------------------------------------------------------------------
void note_launch();        // every kernel launch of the library calls this once
long long launch_count();

// ---- host planner ----------------------------------------------------------------------
int plan_params(int64_t c_cols, int64_t s_lm, const spgemm_options* ov, spgemm_plan* out);
Ladder make_ladder(int64_t tau);

// ---- scans (k_scan.cu) ------------------------------------------------------------------
// out[i] = sum_{j<i} in[j] for i in [0, n]; out has n+1 entries; in may equal out.
// `scratch` holds scan_scratch_elems(n) int64.
int64_t scan_scratch_elems(int64_t n);
void scan_excl_i64(const int64_t* in, int64_t* out, int64_t n, int64_t* scratch, cudaStream_t s);

// ---- setup kernels (k_setup.cu) --------------------------------------------------------
void launch_brow_minmax(const spgemm_csr& B, int32_t* bmin, int32_t* bmax, cudaStream_t s);
void launch_row_ip(const spgemm_csr& A, const spgemm_csr& B, const int32_t* bmin,
                   const int32_t* bmax, const BinRule& rule, int64_t* ip, int32_t* span_lo,
                   uint8_t* bin, cudaStream_t s);
// Stable multisplit of items [0, n) by bin id (bins [0, nbins); kBinEmpty skipped).
// cnt: nbins * ceil(n / 1024) + 1 int64 (scanned in place into offsets).
int64_t bin_blocks(int64_t n);
void launch_bin_count(const uint8_t* bin, int64_t n, int nbins, int64_t* cnt, cudaStream_t s);
void launch_bin_scatter(const uint8_t* bin, int64_t n, int nbins, const int64_t* off,
                        int32_t* out, cudaStream_t s);
void launch_bin_starts(const int64_t* off, int64_t nblk, int nbins, int64_t* starts, cudaStream_t s);
void launch_validate(const spgemm_csr& M, uint32_t* err, cudaStream_t s);
void launch_nnz_bins(const int32_t* rows, int64_t n, const int64_t* row_ptr, const BinRule& rule, uint8_t* bin,
                     cudaStream_t s);

// ---- light rows and chunk accumulators (k_accum.cu) ------------------------------------
// Source of one accumulation: a light row of A*B, or a final chunk of C^_reord.
struct RowJob {
  const int32_t* rows;   // bin list (global row ids)
  int64_t count;
  int64_t slots;         // hash slots (or maximal dense span)
  int tpr;               // threads per row (32 or block size)
  bool dense;
};
struct ChunkSet {        // final chunks of one heavy batch
  const int64_t* start;  // element offset in the C^ buffers
  const int64_t* cnt;    // elements
  const int32_t* row;    // batch-local heavy row
  const int32_t* base;   // first column covered
  int64_t* nnz;          // out (symbolic)
  const int64_t* out;    // in (numeric): offset of the chunk inside its C row
  const int32_t* heavy_rows;  // batch-local row -> global row
  const int32_t* col;    // C^ buffers (both halves)
  const double* val;
};
struct Sink {            // where results go
  int64_t* row_nnz;      // symbolic: count per global row (C.row_ptr before the scan)
  const int64_t* row_ptr;// numeric: C.row_ptr
  int32_t* c_col;
  double* c_val;
  int64_t row_begin, row_end;  // numeric row window; output index 0 = row_ptr[row_begin]
};
struct EstSink {          // estimated workflows (numeric pass run before the row sizes are known)
  const int64_t* cap;      // per global row: output capacity (an estimate, or the IP bound)
  const int64_t* row_tmp;  // per global row: offset of its slot in the temporary output
  int32_t* tmp_col;
  double* tmp_val;
  int64_t* est_nnz;        // out per global row: nnz, or -1 when the row overflowed its capacity
};
// est != null: numeric rows write sorted into their temporary slot and their nnz into
// sink.row_nnz, or mark themselves in est_nnz when they do not fit.
void launch_light(const spgemm_csr& A, const spgemm_csr& B, const int32_t* span_lo,
                  const RowJob& job, bool numeric, const Sink& sink, uint32_t* err,
                  cudaStream_t s, const EstSink* est = nullptr);
void launch_chunks(const ChunkSet& cs, const int32_t* list, int64_t count, int64_t slots, int tpr,
                   bool dense, int64_t dense_width, bool numeric, const Sink& sink,
                   uint32_t* err, cudaStream_t s);
size_t light_smem_bytes(int64_t slots, int tpr, bool dense, bool numeric);
// expand-sort-compact rows of at most esc_max_products() products (k_esc.cu): symbolic writes
// sink.row_nnz, numeric writes the sorted row at its final position
int64_t esc_max_products();
void launch_esc(const spgemm_csr& A, const spgemm_csr& B, const int32_t* rows, int64_t n, bool numeric,
                const Sink& sink, uint32_t* err, cudaStream_t s);

// ---- estimated light-row sizing (k_estimate.cu) ------------------------------------------
bool hll_registers_ok(int m);
// one sketch of m one-byte registers per row of B (out: B.rows * m bytes)
void launch_hll_sketch(const spgemm_csr& B, int m, uint8_t* out, cudaStream_t s);
// capacity of the listed rows of A*B (all rows if rows == nullptr): cap[row] = min(ip[row],
// ceil(coef * estimate)); est_out[i] (optional) = the raw estimate of the i-th listed row
void launch_hll_rows(const spgemm_csr& A, const int32_t* rows, int64_t n, const int64_t* ip, const uint8_t* sk,
                     int m, double coef, int64_t* cap, double* est_out, cudaStream_t s);
// intermediate products of every row of A*B
void launch_row_products(const spgemm_csr& A, const spgemm_csr& B, int64_t* ip, cudaStream_t s);
// bin[i] = ladder level of val[rows[i]]
void launch_val_bins(const int32_t* rows, int64_t n, const int64_t* val, const BinRule& rule, uint8_t* bin,
                     cudaStream_t s);
// bin[i] = 2 if est_nnz[rows[i]] < 0 (the row overflowed its slot), else 1 if its create bin is
// at least wide_from (a block bin), else 0
void launch_overflow_bins(const int32_t* rows, int64_t n, const int64_t* est_nnz, const uint8_t* create_bin,
                          int wide_from, uint8_t* bin, cudaStream_t s);
// dst[rows[i]] = base + off[i]
void launch_scatter_off(const int32_t* rows, int64_t n, const int64_t* off, int64_t base, int64_t* dst,
                        cudaStream_t s);
// listed rows inside [row_begin, row_end): temporary slot -> final position (wide: 32 lanes
// per row, else 8)
void launch_copy_rows(const int32_t* rows, int64_t n, const int64_t* row_tmp, const int64_t* row_ptr,
                      int64_t row_begin, int64_t row_end, const int32_t* tcol, const double* tval, int32_t* ccol,
                      double* cval, bool wide, cudaStream_t s);

// ---- long rows by a shared + global hash (k_long.cu) -------------------------------------------
size_t long_smem_bytes(bool numeric);
int long_blocks(int sms);
// rows[0..nrows) of a group, global table of row j at slots [goff[j] - gbase, goff[j+1] - gbase) of
// gkeys / gvals; gbits: 2 * nwords words per block (numeric); symbolic writes sink.row_nnz
void launch_long(const spgemm_csr& A, const spgemm_csr& B, const int32_t* rows, int64_t nrows, const int64_t* goff,
                 int64_t gbase, int32_t* gkeys, double* gvals, uint32_t* gbits, int64_t nwords, bool numeric,
                 const Sink& sink, int blocks, uint32_t* err, cudaStream_t s);
// cap[j] = global table slots of rows[j]: the power of two >= 2 x (ip[row], or its nnz from row_ptr)
void launch_long_caps(const int32_t* rows, int64_t n, const int64_t* ip, const int64_t* row_ptr, int64_t* cap,
                      cudaStream_t s);

// ---- Markov-clustering step (k_mcl.cu) -----------------------------------------------------
void launch_col_sums(const spgemm_csr& C, double* sums, cudaStream_t s);  // sums zeroed by the caller
void launch_keep_count(const spgemm_csr& C, const double* sums, double thr, int64_t* counts, cudaStream_t s);
void launch_keep_write(const spgemm_csr& C, const double* sums, double thr, const int64_t* out_rp, int32_t* out_col,
                       double* out_val, cudaStream_t s);

// ---- heavy pipeline (k_heavy.cu) ---------------------------------------------------------
void launch_gather_ip(const int32_t* heavy_rows, int64_t nrows, const int64_t* ip, int64_t* out,
                      cudaStream_t s);
void launch_csc_count(const spgemm_csr& A, const int32_t* heavy_rows, int64_t nrows,
                      int32_t* colcnt, cudaStream_t s);
void launch_slice_sizes(const int32_t* colcnt, const spgemm_csr& B, int64_t kcols,
                        int64_t* colptr_sizes, int64_t* slice_sizes, cudaStream_t s);
// csc_col: the column of every CSC entry (the outer product's slice of it)
void launch_csc_scatter(const spgemm_csr& A, const int32_t* heavy_rows, int64_t nrows,
                        int64_t* cursor, int32_t* csc_row, double* csc_val, int32_t* csc_col, cudaStream_t s);
void launch_copy_i64(const int64_t* src, int64_t* dst, int64_t n, cudaStream_t s);
void launch_gather_rows(const int32_t* src, int32_t* io, int64_t n, cudaStream_t s);
void launch_partition(const int64_t* off, int64_t nseg, int64_t total, int64_t tile, int2* part, cudaStream_t s);
void launch_b_chunk_hist(const spgemm_csr& B, const int32_t* colcnt, int shift, int64_t v, int32_t* bh, uint32_t* err,
                         cudaStream_t s);
// counts[r * v + c] = sum of bh[k * v + c] over the entries (r, k) of the heavy rows; hrp is the
// prefix of the heavy rows' lengths (launch_heavy_row_len + scan), entries = hrp[nrows]; counts
// must be zeroed.
void launch_row_chunk_counts(const spgemm_csr& A, const int32_t* rows, int64_t nrows, const int64_t* hrp,
                             int64_t entries, const int32_t* bh, int64_t v, unsigned long long* counts,
                             cudaStream_t s);
void launch_heavy_row_len(const spgemm_csr& A, const int32_t* rows, int64_t nrows, int64_t* len, cudaStream_t s);
// Direct split of level 0: tiles of kOdTile products, each with its first entry of A~_CSC and
// entry count (launch_od_partition), then the outer product writing into C^_reord.
struct OdTile {
  int64_t a_first;
  int64_t nent;
  int32_t s0, s1;  // slices of the tile's first and last product
};
void launch_od_partition(const int64_t* slice_off, int64_t nseg, int64_t total, const int64_t* colptr,
                         const spgemm_csr& B, OdTile* tiles, cudaStream_t s);
void launch_outer_direct(const int64_t* colptr, const int32_t* csc_row, const double* csc_val,
                         const int32_t* csc_col, const int64_t* slice_off, const OdTile* tiles, int64_t total,
                         const spgemm_csr& B, unsigned long long* cursor, int32_t* out_col, double* out_val,
                         bool with_vals, int shift, int64_t nchunks, uint32_t* err, cudaStream_t s);
void launch_outer_product(const int64_t* colptr, const int32_t* csc_row, const double* csc_val,
                          const int32_t* csc_col, const int64_t* slice_off, const int2* part, int64_t total, const spgemm_csr& B,
                          int64_t* row_cursor, int32_t* chat_col, double* chat_val, bool with_vals,
                          unsigned long long* counts, int shift, int64_t nchunks, uint32_t* err, cudaStream_t s);
void launch_histogram(const int64_t* row_ptr, const int2* part, int64_t total, const int32_t* col, int shift,
                      int64_t nchunks, int64_t group_rows, unsigned long long* counts, bool match, int sms,
                      uint32_t* err, cudaStream_t s);
void launch_chunk_partition(const unsigned long long* counts, int64_t n, int64_t tau,
                            uint8_t* bin, cudaStream_t s);
void launch_reord_meta(const unsigned long long* counts, int64_t nrows_in, int64_t nchunks,
                       const int32_t* xmap, const int32_t* in_row, const int32_t* in_base,
                       int64_t width, int64_t* reord_cnt, int32_t* out_row, int32_t* out_base,
                       cudaStream_t s);
void launch_multisplit(const int64_t* row_ptr, const int2* part, int64_t total, const int32_t* in_col,
                       const double* in_val, int shift, int64_t nchunks, int64_t group_rows, const int32_t* xmap,
                       unsigned long long* reord_cursor, int32_t* out_col, double* out_val, bool with_vals, bool match,
                       int sms, uint32_t* err, cudaStream_t s);
// TMA-staged multisplit (k_msplit_tma.cu); returns false when it cannot run (alignment, bins).
bool launch_multisplit_tma(const int64_t* row_ptr, const int2* part, int64_t total, const int32_t* in_col,
                           const double* in_val, int shift, int64_t nchunks, int64_t group_rows, const int32_t* xmap,
                           unsigned long long* cursor, int32_t* out_col, double* out_val, bool with_vals, int sms,
                           uint32_t* err, cudaStream_t s, uint32_t first_spins = 0);
void launch_final_desc(const int64_t* reord_ptr, int64_t q0, int64_t q1, int64_t elem_base,
                       const int32_t* row, const int32_t* base, int64_t* f_start, int64_t* f_cnt,
                       int32_t* f_row, int32_t* f_base, cudaStream_t s);
void launch_chunk_classify(const int64_t* f_cnt, int64_t n, int64_t bitmap_from, const BinRule& rule,
                           uint8_t* bin, cudaStream_t s);
// bitmap-ordered chunk accumulators (k_chunk.cu); mode 0 symbolic, 1 hash numeric, 2 dense numeric
// Shared memory of one chunk group (mode 2: the dense accumulator block).
size_t chunk_smem_bytes(int64_t width, int64_t slots, int mode, bool warp);
void launch_chunk_bitmap(const ChunkSet& cs, const int32_t* list, int64_t count, int64_t width, int mode,
                         int64_t slots, int tpr, const Sink& sink, uint32_t* err, int* counter, double* gacc,
                         cudaStream_t s);
// One chunk of the smallest hash bin, resolved against the numeric sink (cnt < 0: skipped).
struct ChunkDesc {
  int64_t start;     // element offset in the C^ buffers
  int64_t out;       // first output index (relative to the sink's row window)
  int32_t cnt;       // elements
  int32_t expected;  // entries of C (symbolic count)
  int32_t base;      // first column covered
  int32_t pad;
};
constexpr int64_t kWarpChunkMax = 256;        // elements of the largest chunk in the smallest hash bin
constexpr int64_t kBlockChunkMax = 1024;      // and in the next one
// Numeric hash accumulation of a hash bin by persistent groups: warps for the smallest bin (chunks
// of at most kWarpChunkMax elements), 128-thread blocks for the next (at most kBlockChunkMax);
// desc: count scratch descriptors.
void launch_chunk_groups(const ChunkSet& cs, const int32_t* list, int64_t count, int64_t width, bool warps,
                         const Sink& sink, ChunkDesc* desc, uint32_t* err, cudaStream_t s);
constexpr int kChunkHubSlots = 137;           // hub columns of a dense chunk (k_chunk.cu)

// ---- heavy rows without C^ in HBM (k_fused.cu) ----------------------------------------------
constexpr int64_t kFusedMaxChunks = 2048;      // chunks per row the column split of B supports
// Where the generating accumulators read a chunk's products from: row r of A and, for every
// entry (r, k), the chunk-c part of row k of the column-split B.
struct FusedSrc {
  const int64_t* arp;    // A's row pointers and values (the heavy rows' values are read in place)
  const double* aval;
  const int64_t* hrp;    // batch: prefix of the heavy rows' lengths (entry e0 of batch-local row p)
  const int32_t* seg;    // batch: segment table, (v + 1) x E, chunk-major (launch_segtable)
  int64_t E;             // batch: entries of its heavy rows
  const int32_t* bcol;   // B with every row's entries grouped by chunk
  const double* bval;
  int shift;             // log2 of the chunk width
};
// bo and the split entries of the rows of B with colcnt > 0 (bh: their per-chunk counts);
// bs_val null: columns only
void launch_bsplit(const spgemm_csr& B, const int32_t* colcnt, const int32_t* bh, int shift, int64_t v,
                   int32_t* bo, int32_t* bs_col, double* bs_val, uint32_t* err, cudaStream_t s);
// seg[c * E + e] = B_split position of chunk c of the B row of heavy entry e (c = v: the row's end)
// (ecol: E int32 scratch, the A column of every entry)
void launch_segtable(const spgemm_csr& A, const int32_t* rows, int64_t R, const int64_t* hrp, const spgemm_csr& B,
                     const int32_t* bo, int64_t v, int64_t E, int32_t* ecol, int32_t* seg, cudaStream_t s);
// cursor[f_row[q] * v + (f_base[q] >> shift)] = f_start[q]: the direct split's cursors of a batch
// whose descriptors hold the run starts (generated symbolic)
void launch_cursor_from_desc(const int64_t* f_start, const int32_t* f_row, const int32_t* f_base, int64_t n,
                             int64_t v, int shift, int64_t* cursor, cudaStream_t s);
// final chunks of a batch from its level-0 counts, chunk-major (rptr: the counts' exclusive scan,
// the run starts of the numeric expansion, or null)
void launch_fused_desc(const unsigned long long* counts, const int64_t* rptr, int64_t R, int64_t v, int64_t width,
                       int64_t* f_cnt, int32_t* f_row, int32_t* f_base, int64_t* f_start, cudaStream_t s);
// mode 0 symbolic, 1 hash numeric, 2 dense numeric (persistent blocks, counter zeroed here)
void launch_fused_chunks(const FusedSrc& f, const ChunkSet& cs, const int32_t* list, int64_t count, int64_t width,
                         int mode, int64_t slots, int tpr, const Sink& sink, uint32_t* err, int* counter,
                         cudaStream_t s);
void launch_invert(const int32_t* list, int64_t n, int32_t* xmap, cudaStream_t s);
void launch_offset_copy(const int64_t* src, int64_t n, int64_t delta, int64_t* dst, cudaStream_t s);
// out[0] += sum of a[list[i]], out[1] += sum of b[list[i]] for i < n
void launch_list_sums(const int32_t* list, int64_t n, const int64_t* a, const int64_t* b,
                      unsigned long long* out, cudaStream_t s);
void launch_grid_fill(const int32_t* f_row, const int32_t* f_base, const int64_t* f_nnz, int64_t n,
                      int shift_fin, int64_t nfin, int64_t* grid, cudaStream_t s);
void launch_grid_finish(const int64_t* grid_scanned, const int32_t* f_row, const int32_t* f_base,
                        int64_t n, int shift_fin, int64_t nfin, int64_t* f_out, cudaStream_t s);
void launch_row_totals(const int64_t* grid_scanned, int64_t nrows, int64_t nfin,
                       const int32_t* heavy_rows, int64_t* row_nnz, cudaStream_t s);

}  // namespace sg

// ---- the handle ---------------------------------------------------------------------------
struct LevelInfo {
  int64_t nin = 0;       // input rows of the level
  int64_t v = 0;         // chunks per input row
  int64_t width = 0;     // columns per output chunk
  int64_t nheavy = 0;    // output chunks passed to the next level (heavy ones, stored first)
  int64_t desc0 = 0;     // first final-chunk descriptor written by this level
  int64_t elem_base = 0; // offset of the level's output half in the C^ buffer
  int64_t next_elems = 0;// elements of the heavy chunks (the next level's input)
};

struct HeavyBatch {
  int64_t h0 = 0, h1 = 0;       // range of the heavy-row list
  int64_t row_lo = 0, row_hi = 0;  // smallest and largest global row of the batch
  int64_t elems = 0;            // intermediate products of the batch
  std::vector<LevelInfo> lv;    // recorded by the symbolic phase, replayed by the numeric one
  int64_t nfinal = 0;           // final chunks (C^_reord rows that are accumulated)
  int64_t* f_start = nullptr;
  int64_t* f_cnt = nullptr;
  int32_t* f_row = nullptr;
  int32_t* f_base = nullptr;
  int64_t* f_nnz = nullptr;
  int64_t* f_out = nullptr;
  int32_t* f_list = nullptr;    // chunk ids ordered by accumulator bin
  std::vector<int64_t> f_bin_start;  // host, per chunk bin (size nbins + 1)
  int64_t nnz_c = 0;            // entries of C in the batch's rows (read after the symbolic sync)
  int64_t bitmap_from = 0;      // descriptors from here on are last-level chunks (width W)
  int64_t dense_sums[2] = {0, 0};  // elements and nnz of the chunks on the dense accumulator
  int64_t* f_hrp = nullptr;     // generated products (SPGEMM_FLAG_FUSED): prefix of the rows' lengths
  int64_t entries = 0;          // and the entries of the batch's heavy rows
};

struct spgemm_ctx {
  int64_t m = 0, k = 0, n = 0;
  spgemm_csr A{}, B{};
  cudaStream_t st = nullptr;
  cudaStream_t st_light = nullptr;  // light rows (the heavy pipeline stays on st)
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  cudaStream_t st_copy = nullptr;   // device-to-host copies of the host-streamed numeric phase
  cudaEvent_t ev_done[2] = {nullptr, nullptr}, ev_copied[2] = {nullptr, nullptr};
  int device = 0, sms = 0;
  cudaMemPool_t pool = nullptr;
  int64_t smem_optin = 0, l2_bytes = 0;
  spgemm_options opt{};
  spgemm_plan plan{};
  sg::Ladder lad;
  sg::BinRule rule{};
  int nbins = 0;                // 2 * ladder levels + 1 (heavy)
  spgemm_stats stats{};
  int state = 0;                // 1 after create, 2 after symbolic
  int64_t* c_row_ptr = nullptr; // remembered from symbolic

  // workspace (device)
  std::vector<void*> allocs;
  std::vector<size_t> alloc_bytes;  // sizes of allocs (the workspace budget counts them)
  size_t ws_bytes = 0;              // live workspace bytes
  uint32_t* d_err = nullptr;
  int* d_counter = nullptr;     // work counter of the persistent dense accumulator
  double* d_gacc = nullptr;     // L2-resident dense accumulators (SPGEMM_FLAG_DENSE_L2)
  int64_t* d_scan = nullptr;    // scan scratch
  int64_t scan_cap = 0;
  int64_t* d_ip = nullptr;
  int32_t* d_span_lo = nullptr;
  uint8_t* d_bin = nullptr;
  int32_t* d_rows = nullptr;    // concatenated stable bin lists
  int64_t* d_binoff = nullptr;
  std::vector<int64_t> bin_start;  // host copy (nbins + 1)
  // numeric-phase bins of the light hash rows, by their exact size (built on the first numeric call)
  int32_t* d_nrows = nullptr;
  std::vector<int64_t> nbin_start;

  // heavy rows
  int64_t nheavy = 0;
  const int32_t* d_heavy = nullptr;   // into d_rows
  int64_t* d_heavy_pre = nullptr;     // exclusive prefix of heavy IP (nheavy + 1)
  std::vector<int64_t> heavy_pre;     // host copy
  std::vector<HeavyBatch> batches;
  int64_t batch_cap = 0;              // elements per C^ buffer
  int32_t* d_chat_col = nullptr;      // 2 * batch_cap (ping-pong halves)
  double* d_chat_val = nullptr;
  bool resident = false;
  bool chat_has_vals = false;

  // phase timing (slots: see spgemm_get_phase_times)
  bool timing = false;

  // numeric phase replayed from a CUDA graph: captured on the second call with the same row
  // range and output arrays, when that phase enqueues no host synchronisation and no allocation
  cudaGraphExec_t num_exec = nullptr;
  cudaStream_t st_graph = nullptr;  // capture stream (the caller's may be the legacy default stream)
  int64_t num_rb = -1, num_re = -1;
  int32_t* num_col = nullptr;
  double* num_val = nullptr;
  int num_calls = 0;           // eager calls with the current key
  long long num_launches = 0;  // kernel launches the graph holds
  bool capturing = false;      // ws_alloc refuses while a capture is open
  bool last_graph = false;     // the last numeric call ran from the graph

  int esc_levels = 0;           // ladder levels whose light rows take the ESC accumulator

  // heavy rows without C^ (SPGEMM_FLAG_FUSED): the column split of B, kept between the phases
  bool fused = false;
  int32_t* d_colcnt = nullptr;  // per row of B: entries of heavy rows of A that use it
  int32_t* d_bh = nullptr;      // B.rows x v: entries of row k in chunk c
  int32_t* d_bo = nullptr;      // B.rows x (v + 1): offsets of the chunks inside row k
  int32_t* d_bs_col = nullptr;  // B's entries grouped by chunk inside every row
  double* d_bs_val = nullptr;
  bool long_rows = false;       // heavy rows by the shared + global hash (SPGEMM_FLAG_LONG_ROWS)
  bool gen_symbolic = false;    // symbolic by generated products, numeric by the direct split
  sg::ChunkDesc* d_cdesc = nullptr;  // descriptors of the smallest numeric hash bin (largest batch)
  int64_t cdesc_cap = 0;
  int32_t* d_seg = nullptr;     // segment table of the batch being accumulated (launch_segtable)
  int64_t seg_cap = 0;
  int32_t* d_ecol = nullptr;    // the A column of each of its entries
  int64_t ecol_cap = 0;

  // light rows sized by their IP bound or by HyperLogLog estimates (SPGEMM_WORKFLOW_*)
  int workflow = 0;            // the workflow the symbolic phase ran
  int hll_m = 0;               // registers per sketch
  double hll_coef = 0.0;
  uint8_t* d_sketch = nullptr; // one sketch per row of B
  int64_t* d_cap = nullptr;    // per row: capacity of its temporary slot
  int64_t* d_row_tmp = nullptr;// per row: offset of its slot
  int64_t* d_est_nnz = nullptr;// per row: nnz, or -1 (overflowed)
  int32_t* d_tmp_col[2] = {nullptr, nullptr};  // temporary output: first pass, fallback pass
  double* d_tmp_val[2] = {nullptr, nullptr};
  // rows to copy out: rows of the warp bins and of the block bins from the first temporary
  // output, the fallback rows from the second
  const int32_t* d_est_list[3] = {nullptr, nullptr, nullptr};
  int64_t est_count[3] = {0, 0, 0};
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> timed[sg::kPhaseSlots];
  double phase_ms[sg::kPhaseSlots] = {0};
  int64_t phase_n[sg::kPhaseSlots] = {0};
};

namespace sg {
// api.cu helpers used by the heavy orchestration
void* ws_alloc(spgemm_ctx* h, size_t bytes);
void ws_free(spgemm_ctx* h, void* p);
int check_cuda(cudaError_t e, const char* what);
void set_last_error(const std::string& s);
}  // namespace sg
