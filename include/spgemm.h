/*
 * spgemm.h -- C ABI of libspgemm_gb300.so: single-GPU sparse general matrix-matrix product
 * C = A * B on CSR matrices (int64 row pointers, int32 column indices, fp64 values), for
 * NVIDIA GB300 (sm_103a).
 *
 * The method is the gMAGNUS pipeline ("gMAGNUS: Fast SpGEMM on GPUs for Irregular Matrices
 * via Hierarchical Multisplit", arXiv 2607.22866v1):
 *   - per-row intermediate-product (IP) count and light/heavy partition (section III-A,
 *     Algorithm 3, setup phase);
 *   - light rows: Gustavson row-wise accumulation in shared-memory hash maps, or in a
 *     shortened dense accumulator when the row's column span is narrow (section II-B,
 *     section III-E; bin ladder after "Ocean: Fast Estimation-Based SpGEMM on GPU",
 *     section 4, kernel configurations);
 *   - heavy rows: masked CSR-to-CSC of A, outer-product expansion into an intermediate
 *     matrix C^ (section III-B, Algorithm 4), hierarchical histogram + multisplit by column
 *     range into C^_reord (section III-C, Algorithm 5), chunk accumulation in shared memory
 *     (section III-E) written straight to the final CSR positions;
 *   - an exact symbolic phase that sizes C.row_ptr through a device scan, then a numeric
 *     phase (section II-B, Algorithm 1 and the symbolic/numeric split).
 *
 * Conventions for every entry point:
 *   - Return value: SPGEMM_OK (0) or one of the negative codes below; spgemm_strerror()
 *     names it and spgemm_last_error() gives a one-line detail for the calling thread.
 *   - "device" pointers point into the current CUDA device's global memory; "host" pointers
 *     into ordinary process memory.  The library never frees a pointer it did not allocate.
 *   - All GPU work is ordered on the stream given to spgemm_create (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  Calls return once the work is enqueued,
 *     except where a host result is returned (noted below), which synchronises that stream.
 *   - A handle is not thread-safe: use one handle per host thread.
 *   - Failure of a device-side check (hash probe limit, inconsistent input) is reported as
 *     SPGEMM_ERR_DEVICE at the next synchronising call; kernels never trap.
 */
#ifndef SPGEMM_GB300_H
#define SPGEMM_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------------------ */
#define SPGEMM_OK 0
#define SPGEMM_ERR_INVALID_ARG (-1)  /* null pointer, negative size, shape mismatch        */
#define SPGEMM_ERR_INVALID_CSR (-2)  /* optional validation: row_ptr / col_idx malformed    */
#define SPGEMM_ERR_BAD_STATE (-3)    /* call out of order (numeric before symbolic, ...)    */
#define SPGEMM_ERR_OUT_OF_MEMORY (-4)/* workspace allocation failed                          */
#define SPGEMM_ERR_OVERFLOW (-5)     /* a size does not fit the index types (C.cols > 2^31-1) */
#define SPGEMM_ERR_DEVICE (-6)       /* a kernel reported an internal check failure          */
#define SPGEMM_ERR_CUDA (-7)         /* a CUDA runtime call failed (detail in last_error)    */

/* ---- option flags (spgemm_options.flags) ------------------------------------------ */
#define SPGEMM_FLAG_ALL_HEAVY 1       /* route every non-empty row through the heavy path   */
#define SPGEMM_FLAG_ALL_LIGHT 2       /* keep every row with IP <= tau light even when ALL_HEAVY is
                                         set; rows above tau are always heavy (no light table fits) */
#define SPGEMM_FLAG_NO_DENSE_LIGHT 4  /* light rows never use the shortened dense accumulator */
#define SPGEMM_FLAG_VALIDATE 8        /* check A and B (row_ptr monotone, columns in range)  */
#define SPGEMM_FLAG_RECOMPUTE 16      /* never keep C^_reord between symbolic and numeric    */
#define SPGEMM_FLAG_TIMING 32         /* record device time per phase (CUDA events, no syncs) */
#define SPGEMM_FLAG_NO_MATCH 64       /* multisplit: plain shared atomics instead of
                                         __match_any_sync warp aggregation */
#define SPGEMM_FLAG_DENSE_L2 128      /* heavy dense chunks sum with L2 reductions into a global
                                         per-SM array instead of shared-memory atomics */
#define SPGEMM_FLAG_TMA_SPLIT 512     /* multisplit: tiles of C^ staged in shared memory by
                                         bulk copies (two stages per block) instead of held in
                                         registers; slower on the R-MAT cases */
#define SPGEMM_FLAG_FUSED_HIST 1024   /* level-0 histogram counted per product inside the outer
                                         product (warp match + global atomics) instead of from
                                         per-B-row chunk counts summed over the rows of A */
#define SPGEMM_FLAG_DIRECT_SPLIT 256  /* one-level plans: the outer product writes straight into
                                         C^_reord (counts from per-B-row chunk histograms), so C^
                                         is never stored and level 0 needs no multisplit pass.
                                         The default since it measured faster; kept for callers
                                         that set it */
#define SPGEMM_FLAG_EXPAND_SPLIT 16384 /* one-level plans too: the outer product writes C^ and a
                                         separate multisplit pass builds C^_reord (the paper's
                                         flow; also taken with NO_MATCH, TMA_SPLIT or FUSED_HIST) */
#define SPGEMM_FLAG_NO_GRAPH 2048    /* never capture or replay the numeric phase as a CUDA graph */
#define SPGEMM_FLAG_FUSED 8192       /* heavy rows without the intermediate matrix in HBM: the
                                        rows of B are split once by column chunk, and every
                                        (heavy row, chunk) accumulator generates its own products
                                        from A and the split B instead of reading them from
                                        C^_reord (no outer product, no multisplit pass, no heavy
                                        batches to recompute); taken when a row has at most 2048
                                        chunks and B has fewer than 2^31 entries (stats.fused) */
#define SPGEMM_FLAG_LONG_ROWS 32768  /* heavy rows by a long-row hash accumulator instead of the
                                        outer product + multisplit + chunk accumulators: one block
                                        per row, a shared-memory table that spills into a global
                                        table of the row, output ordered by a bitmap of the row's
                                        columns (after the Ocean page's hybrid accumulator for
                                        long rows; stats.long_rows) */
#define SPGEMM_FLAG_NO_GEN_SYMBOLIC 65536 /* products whose heavy expansion is recomputed in the
                                        numeric phase (stats.resident == 0) count their heavy
                                        chunks in the symbolic phase from products generated out of
                                        the column-split B, not from an expansion of the columns;
                                        this flag keeps the column expansion (stats.gen_symbolic) */
#define SPGEMM_FLAG_HASH_PER_CHUNK 131072 /* numeric heavy chunks of at most 1024 elements: a warp
                                        (at most 256 elements) or a block per chunk that clears its
                                        table and bitmap first, instead of the default persistent
                                        warps and blocks whose tables are sized to each chunk and
                                        emptied by their final sweep */
#define SPGEMM_FLAG_NO_ESC 4096      /* light hash rows with at most 64 intermediate products
                                        use the shared-memory hash table like longer rows, instead
                                        of the default expand-sort-compact accumulator held in one
                                        warp's registers (exact symbolic workflow; narrow rows
                                        always take the shortened dense accumulator) */

/* A CSR matrix in device memory, borrowed by the library (never written or freed). */
typedef struct {
  int64_t rows, cols, nnz;
  const int64_t* row_ptr; /* device, rows+1 entries, row_ptr[0] = 0, non-decreasing, row_ptr[rows] = nnz */
  const int32_t* col_idx; /* device, nnz entries, 0 <= col < cols; rows need not be sorted; repeats are separate terms */
  const double* vals;     /* device, nnz entries */
} spgemm_csr;

/* Planner overrides; a zero field means "derive from the device".  Used by tests (to force
 * several multisplit levels and both paths on tiny inputs) and for tuning. */
typedef struct {
  int64_t tau;               /* heavy threshold: rows (and chunks) with more IP are heavy */
  int64_t chunk_width;       /* dense accumulator width W of the last level (power of two) */
  int64_t chunks_max;        /* most chunks one multisplit level may create (power of two) */
  int64_t heavy_batch_elems; /* most heavy intermediate products expanded at once          */
  int64_t smem_bytes;        /* shared-memory budget s_LM per thread block                 */
  int32_t flags;             /* SPGEMM_FLAG_* */
  int32_t workflow;          /* SPGEMM_WORKFLOW_*: how the light rows are sized (0: exact symbolic) */
  int32_t hll_registers;     /* estimated workflow: 32 or 64 registers per sketch (0: by the
                                expansion ratio, 32 below 48 products per entry of A, else 64) */
  int32_t reserved;
  double hll_coef;           /* estimated workflow: capacity = ceil(coef * estimate) (0: 2.0 with
                                32 registers, 1.5 with 64) */
  int64_t workspace_limit;   /* most bytes of device workspace the handle may hold at once (0: no
                                limit); an allocation past it fails with SPGEMM_ERR_OUT_OF_MEMORY */
  int32_t debug_hash_slots;  /* tests: cap every light-row hash table at this many slots (0: off), so
                                that longer rows overflow their table (SPGEMM_ERR_DEVICE) */
  int32_t debug_wait_spins;  /* tests: polls allowed to the first bulk-copy wait of every block of the
                                staged multisplit (SPGEMM_FLAG_TMA_SPLIT; 0: the normal limit), so that
                                a test reaches its timeout path (SPGEMM_ERR_DEVICE) */
} spgemm_options;

/* Light-row sizing (Ocean page, Table 1 and the estimation-based workflow).  SYMBOLIC counts
 * every light row exactly before the numeric phase.  UPPER_BOUND and ESTIMATE skip that count:
 * the light rows are accumulated during spgemm_symbolic into temporary slots of a capacity --
 * the row's intermediate-product count (a bound), or a HyperLogLog estimate times a coefficient
 * -- and their exact sizes come out of that pass; rows that do not fit their estimated slot are
 * accumulated again with the bound.  spgemm_numeric then copies them to their final positions.
 * The light rows' values are therefore read during spgemm_symbolic.  AUTO applies the page's
 * selection: UPPER_BOUND when the average row has fewer than 64 intermediate products, ESTIMATE
 * when the expansion ratio (products per entry of A) and the sampled compression ratio
 * (products per entry of C, from HyperLogLog estimates of 3% of the light rows, 600 to 10,000) are
 * both at least 8, else SYMBOLIC.  Heavy rows always take the exact multisplit path. */
#define SPGEMM_WORKFLOW_SYMBOLIC 0
#define SPGEMM_WORKFLOW_UPPER_BOUND 1
#define SPGEMM_WORKFLOW_ESTIMATE 2
#define SPGEMM_WORKFLOW_AUTO 3

#define SPGEMM_MAX_LEVELS 8

/* Parameters of the gMAGNUS planner (gMAGNUS page, section III-D, Eq. (4)-(7)). */
typedef struct {
  int64_t s_lm;              /* shared-memory bytes per block the accumulators may use      */
  int64_t tau;               /* heavy threshold, Eq. (4): s_LM / (alpha * (s_col + s_val)), alpha = 2 */
  int64_t dense_numeric;     /* n_denseNumeric = s_LM / (s_val + s_bitmap), bitmap = 1/8 byte */
  int64_t chunk_width;       /* W: dense_numeric floored to a power of two (or override)    */
  int64_t chunks_required;   /* ceil(C.cols / W) rounded up to a power of two                */
  int64_t chunks_max;        /* Eq. (6) for this build's multisplit kernel, floored to pow2  */
  int32_t levels;            /* Eq. (7): ceil(log2(required) / log2(max)), 1 if required <= max */
  int32_t reserved;
  int64_t v_chunks[SPGEMM_MAX_LEVELS]; /* chunks per row per level: max, ..., required / max^(levels-1) */
  int64_t group_elems_op;    /* flattened elements per outer-product thread block            */
  int64_t group_elems_ms;    /* flattened elements per histogram / multisplit thread block   */
  int64_t group_rows;        /* n_groupRows = ceil((group_elems_ms - 1) / tau) + 1           */
} spgemm_plan;

/* Counters of one product, filled after spgemm_create / spgemm_symbolic. */
typedef struct {
  int64_t m, k, n;
  int64_t ip_total;          /* intermediate products of all rows                      */
  int64_t ip_heavy;          /* of heavy rows                                           */
  int64_t rows_heavy, rows_light, rows_empty;
  int64_t rows_dense_light;  /* light rows on the shortened dense accumulator           */
  int64_t c_nnz;             /* -1 before spgemm_symbolic                               */
  int64_t heavy_batches;     /* expansions of heavy rows per phase                      */
  int64_t levels_run;        /* multisplit levels executed (<= plan.levels)             */
  int64_t final_chunks;      /* C^_reord rows accumulated                               */
  int64_t chunks_dense;      /* of which on the dense accumulator                       */
  int64_t chat_bytes;        /* bytes of C^ col+val per batch buffer (largest batch)    */
  int64_t c_nnz_heavy;       /* entries of C in heavy rows (after spgemm_symbolic)      */
  int64_t dense_elems;       /* C^_reord elements summed on the dense accumulator       */
  int64_t dense_nnz;         /* entries of C those dense chunks produce                 */
  int32_t resident;          /* 1: C^_reord kept from symbolic to numeric               */
  int32_t numeric_graph;     /* 1: the last numeric call replayed a captured CUDA graph */
  int64_t rows_overflow;     /* estimated workflow: light rows that exceeded their slot    */
  int32_t workflow;          /* SPGEMM_WORKFLOW_* the symbolic phase ran (after AUTO)      */
  int32_t hll_registers;     /* registers per sketch (estimated workflow), else 0          */
  int32_t fused;             /* 1: heavy rows generated their products (SPGEMM_FLAG_FUSED)  */
  int32_t direct_split;      /* 1: level 0 split inside the outer product (one-level plans)  */
  int32_t long_rows;         /* 1: heavy rows by the long-row hash (SPGEMM_FLAG_LONG_ROWS)   */
  int32_t gen_symbolic;      /* 1: heavy chunks counted from generated products in symbolic */
} spgemm_stats;

typedef struct spgemm_ctx* spgemm_handle;

/* Planner alone (host only, no GPU).  c_cols = C.cols; s_lm = shared-memory bytes per block
 * (opt-in maximum on the device); ov may be NULL.  Fills *out.  gMAGNUS page, section
 * III-D.  Returns SPGEMM_ERR_INVALID_ARG for c_cols < 0, s_lm < 4096, or overrides that are
 * not powers of two. */
int spgemm_plan_params(int64_t c_cols, int64_t s_lm, const spgemm_options* ov, spgemm_plan* out);

/* Start a product C = A * B with A m-by-k and B k-by-n.  Borrows A and B (device CSR), which
 * must stay valid and unchanged until spgemm_destroy.  Runs the setup phase (gMAGNUS page,
 * Algorithm 3, setup part: planner, IP per row, partition and binning) and synchronises the
 * stream once to read the bin sizes.  On success *h owns its device workspace.  stream is a
 * cudaStream_t.  Errors: INVALID_ARG (null pointers, A.cols != k, B.rows != k, negative or
 * inconsistent sizes), OVERFLOW (n > 2^31-1), INVALID_CSR (with SPGEMM_FLAG_VALIDATE),
 * OUT_OF_MEMORY, CUDA. */
int spgemm_create(spgemm_handle* h, int64_t m, int64_t k, int64_t n, const spgemm_csr* A,
                  const spgemm_csr* B, void* stream);
int spgemm_create_ex(spgemm_handle* h, int64_t m, int64_t k, int64_t n, const spgemm_csr* A,
                     const spgemm_csr* B, void* stream, const spgemm_options* opt);

/* Symbolic phase: writes C.row_ptr (device, m+1 int64, caller-owned) and *c_nnz (host).
 * Row i of C holds every column that receives at least one product, including sums that are
 * exactly zero.  Synchronises the stream.  May be called once per handle. */
int spgemm_symbolic(spgemm_handle h, int64_t* c_row_ptr, int64_t* c_nnz);

/* Numeric phase: writes C.col_idx (device, c_nnz int32) and C.vals (device, c_nnz fp64),
 * caller-owned, each row sorted by column, at the positions of the row_ptr from
 * spgemm_symbolic (which must still hold those values).  May be called more than once.  When
 * no C^_reord is kept from symbolic (stats.resident == 0: no heavy row, or SPGEMM_FLAG_RECOMPUTE)
 * and the light rows were sized exactly (stats.workflow == SPGEMM_WORKFLOW_SYMBOLIC), every call
 * reads the current values of A and B, so their values (never their structure) may change
 * between calls.  A call repeating the previous one's arguments is captured into a CUDA
 * graph, and later repeats replay it (stats.numeric_graph), when the phase needs no host
 * synchronisation: no heavy row, or C^_reord resident.  SPGEMM_FLAG_NO_GRAPH turns this off. */
int spgemm_numeric(spgemm_handle h, int32_t* c_col_idx, double* c_vals);

/* Numeric phase for rows [row_begin, row_end) only, written at offset 0 = row_ptr[row_begin]
 * of the given arrays (which need row_ptr[row_end] - row_ptr[row_begin] entries).  Lets a
 * caller stream a C too large for the device in row blocks. */
int spgemm_numeric_rows(spgemm_handle h, int64_t row_begin, int64_t row_end, int32_t* c_col_idx,
                        double* c_vals);

/* Numeric phase into HOST memory: c_col_idx (c_nnz int32) and c_vals (c_nnz fp64) are host
 * arrays, caller-owned (page-locked memory reaches the full copy bandwidth; pageable memory
 * works, slowly).  C is computed in row windows of about window_nnz entries (0: a quarter of
 * C, at least 4 M entries, staging at most a fifth of the free device memory) into two device
 * staging buffers from the handle's pool; each finished window is copied to the host on a
 * second stream while the next one is computed.  When heavy batches are recomputed in the
 * numeric phase, windows hold whole batches.  If c_row_ptr is not NULL it receives the m+1
 * row offsets (host).  Returns after every copy has landed; no device array of C's size is
 * needed, so a C larger than the device can be produced.  Errors: BAD_STATE before symbolic,
 * INVALID_ARG for NULL arrays with c_nnz > 0 or a negative window, OUT_OF_MEMORY when a
 * window's staging does not fit.  The pages have no counterpart: it is the host end of the
 * row-window numeric phase. */
int spgemm_numeric_host(spgemm_handle h, int64_t* c_row_ptr, int32_t* c_col_idx, double* c_vals,
                        int64_t window_nnz);

/* Row windows for a numeric phase run window by window (spgemm_numeric_rows into one reused
 * buffer, for a C larger than the device).  Windows cover [0, m) in order; each holds about
 * target_nnz entries of C (0: a quarter of C, at least 4 M entries).  When the heavy rows'
 * expansion is recomputed in the numeric phase (stats.resident == 0 with several heavy
 * batches), every cut falls between two heavy batches, so each batch is expanded once per
 * pass over the windows; such windows may hold more than target_nnz entries.
 *   cuts:           host, cap int64 entries; receives n_windows + 1 row indices, cuts[0] = 0,
 *                   cuts[n_windows] = m, window w = rows [cuts[w], cuts[w+1]);
 *   n_windows:      host, receives the number of windows (also when cap is too small);
 *   max_window_nnz: host (may be NULL), receives the entries of C in the largest window.
 * Copies C.row_ptr to the host and synchronises the stream.  Errors: BAD_STATE before
 * spgemm_symbolic; INVALID_ARG for NULL pointers, negative sizes, or cap < n_windows + 1
 * (n_windows and max_window_nnz are set, so the caller can retry with a longer array).  The
 * pages have no counterpart: it serves the row-window numeric phase. */
int spgemm_row_windows(spgemm_handle h, int64_t target_nnz, int64_t* cuts, int64_t cap, int64_t* n_windows,
                       int64_t* max_window_nnz);

int spgemm_get_stats(spgemm_handle h, spgemm_stats* out);
int spgemm_get_plan(spgemm_handle h, spgemm_plan* out);

/* Cumulative device time (milliseconds, CUDA events recorded on the handle's stream around
 * every timed region) and number of timed regions per slot, since create:
 *   0 setup, 1 light symbolic, 2 masked CSR-to-CSC + slice offsets, 3 outer-product kernel,
 *   4 histogram kernel, 5 multisplit kernel, 6 multisplit bookkeeping (partition, offsets),
 *   7 heavy chunk symbolic, 8 chunk offsets, 9 C.row_ptr scan, 10 light numeric,
 *   11 heavy chunk numeric (all chunk kernels), 12 its dense-accumulator kernel alone.
 * Only recorded when the handle was created with SPGEMM_FLAG_TIMING or the environment
 * variable SPGEMM_TIMING=1.  Synchronises the stream.  t and launches (may be NULL) receive
 * min(count, 13) entries. */
int spgemm_get_phase_times(spgemm_handle h, double* t, int64_t* launches, int32_t count);

/* Number of kernels this library has launched in the process so far (all handles). */
long long spgemm_kernel_launches(void);

/* Device workspace comes from a stream-ordered memory pool (one per device) that keeps freed
 * memory cached for the next product, and the library's internal streams and events are kept
 * for reuse by later handles.  This returns the cached memory to the device and destroys the
 * kept streams and events; call it when no product is running (and before any device reset).
 * Always SPGEMM_OK. */
int spgemm_release_memory(void);

/* Release the workspace (stream-ordered on the handle's stream) and the handle.  NULL is ok. */
int spgemm_destroy(spgemm_handle h);

/* HyperLogLog output-size estimates for every row of C = A * B (Ocean page: HyperLogLog
 * background, construct-and-merge of Figure 3).  One sketch of `registers` (32 or 64) one-byte
 * registers per row of B: a column's 32-bit hash (MurmurHash3 finaliser) picks its register by
 * the low bits and offers 1 + the leading zeros of the other bits; row i's sketch is the
 * element-wise maximum over the rows of B that row i of A selects; its estimate is the
 * HyperLogLog harmonic-mean estimate with linear counting below 5m/2.  Writes cap[i] =
 * min(IP_i, ceil(coef * estimate_i)) (0 for rows without products) into the DEVICE array cap (A.rows
 * int64).  A and B are device CSR with A.cols == B.rows.  Enqueued on `stream`; scratch is
 * allocated and freed stream-ordered.  Errors: INVALID_ARG (null pointers, shape mismatch,
 * registers not 32 or 64, coef <= 0), OUT_OF_MEMORY, CUDA. */
int spgemm_hll_estimate(const spgemm_csr* A, const spgemm_csr* B, int32_t registers, double coef,
                        int64_t* cap, void* stream);

/* Markov-clustering step after the expansion C = M * M (Trident page, section 5.7): normalize
 * the columns of C, prune the entries below `threshold`, square the remaining entries.  An
 * entry (i, j) is kept when C[i,j] / colsum_j >= threshold; its new value is
 * (C[i,j] / colsum_j)^2; rows keep C's column order.  C is device CSR (any row order inside
 * rows).  Symbolic part: writes col_sums (device, C.cols doubles; fp64 sums, order not fixed),
 * out_row_ptr (device, C.rows + 1) and *out_nnz (host); synchronises `stream`.  Numeric part:
 * writes out_col / out_val (device, *out_nnz entries, caller-owned) at out_row_ptr, using the
 * col_sums of the symbolic part.  Errors: INVALID_ARG (null pointers, threshold < 0),
 * OUT_OF_MEMORY (scan scratch), CUDA. */
int spgemm_mcl_prune_symbolic(const spgemm_csr* C, double threshold, double* col_sums, int64_t* out_row_ptr,
                              int64_t* out_nnz, void* stream);
int spgemm_mcl_prune_numeric(const spgemm_csr* C, double threshold, const double* col_sums,
                             const int64_t* out_row_ptr, int32_t* out_col, double* out_val, void* stream);

/* C.row_ptr and nnz(C) without allocating any device memory.  The paper has no counterpart:
 * this entry point exists for callers that cannot call cudaMalloc (or any allocator) at the
 * point where they need the row sizes of C -- code running inside an allocator or memory
 * manager, loops that forbid allocation after start-up, hosts with a fixed memory budget.
 * Instead of a workspace it uses one static __device__ array of 33,280 bytes that every
 * device which loads this library holds until the process exits.
 *   m, k, n, A, B: as for spgemm_create (A and B in device memory, borrowed);
 *   c_row_ptr:     device, m+1 int64, caller-owned, written with the exclusive scan of the
 *                  distinct column counts of the rows of A*B (identical to spgemm_symbolic);
 *   c_nnz:         host, receives nnz(C);
 *   stream:        cudaStream_t; the call synchronises it before returning.
 * Limits: m <= 16,777,215 rows and at most 2048 intermediate products in every row of A*B.
 * Errors: INVALID_ARG for null pointers, mismatched shapes, more rows than the limit, a row
 * above the product limit or a row pointer / column index out of range (the last two are
 * detected on the device after the kernels ran; c_row_ptr is then meaningless); DEVICE when a
 * row's hash table filled up (not expected within the limits); OVERFLOW for k or n above
 * 2^31-1; CUDA for a failed runtime call.  No cudaMalloc, cudaFree or allocating library call
 * is made by the call itself.  With CUDA's lazy module loading, though, the first call on a
 * device loads this code and its static array into that device's memory and looks up the
 * array's address (cudaGetSymbolAddress, with that device current): make one warm-up call per
 * device at start-up (m = 0 is enough), before any stream capture and before entering code
 * that must not allocate.  Every call on a device shares the one array: calls that overlap on
 * the GPU (other streams, other host threads) race and give wrong results; serialise them. */
int spgemm_symbolic_noalloc(int64_t m, int64_t k, int64_t n, const spgemm_csr* A,
                            const spgemm_csr* B, int64_t* c_row_ptr, int64_t* c_nnz, void* stream);

const char* spgemm_strerror(int code);
/* Detail of the last failure on the calling host thread ("" if none). */
const char* spgemm_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SPGEMM_GB300_H */
