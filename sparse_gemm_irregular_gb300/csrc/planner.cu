// Host planner: the gMAGNUS parameters (gMAGNUS page, section III-D, Eq. (4)-(7)).
//
// Readings of the page taken here (the printed formulas are partly garbled):
//  * Eq. (4) prints tau = s_LM / ((1/alpha) * s_col * s_val); the text around it describes a
//    hash map of capacity tau at load factor 1/alpha holding (col, val) pairs, so
//    tau = s_LM / (alpha * (s_col + s_val)) with alpha = 2.
//  * The last level's chunk count is printed as n_required - n_max^(levels-1); Tables V and
//    VI of the same page (e.g. "128: 64, 2", "4096: 32, 32, 4") show a quotient, so
//    v_chunks[last] = n_required / n_max^(levels-1).
//  * The dense width is floored to a power of two; the required chunk count is rounded up to
//    a power of two (the only rounding that reproduces every "Num. Chunks" cell), and one
//    level suffices when n_required <= n_max (PVC soc-Slashdot0902: 32 with a maximum of 32).
//  * Eq. (6) is evaluated with this build's multisplit kernel: one block-wide histogram with
//    warp-aggregated updates (n_subGroups = 1) whose entries carry a 4-byte count and a 4-byte
//    local offset (s_histo = 8), an 8-byte global offset per bin (s_rowPtr), and a fixed
//    element tile per block (n_minGroupElems) held in registers and shared memory.
#include <string.h>

#include "internal.h"

namespace sg {

static bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }
static int64_t floor_pow2(int64_t x) {
  int64_t p = 1;
  while (p * 2 <= x) p *= 2;
  return p;
}
static int64_t ceil_pow2(int64_t x) {
  int64_t p = 1;
  while (p < x) p *= 2;
  return p;
}

int plan_params(int64_t c_cols, int64_t s_lm, const spgemm_options* ov, spgemm_plan* out) {
  if (!out || c_cols < 0 || s_lm < 4096) return SPGEMM_ERR_INVALID_ARG;
  spgemm_options o;
  memset(&o, 0, sizeof(o));
  if (ov) o = *ov;
  if (o.tau < 0 || o.chunk_width < 0 || o.chunks_max < 0 || o.heavy_batch_elems < 0)
    return SPGEMM_ERR_INVALID_ARG;
  if (o.chunk_width && !is_pow2(o.chunk_width)) return SPGEMM_ERR_INVALID_ARG;
  if (o.chunks_max && (!is_pow2(o.chunks_max) || o.chunks_max < 2)) return SPGEMM_ERR_INVALID_ARG;

  spgemm_plan p;
  memset(&p, 0, sizeof(p));
  p.s_lm = s_lm;
  const int64_t s_col = 4, s_val = 8, alpha = 2;
  p.tau = o.tau ? o.tau : s_lm / (alpha * (s_col + s_val));
  p.dense_numeric = (s_lm * 8) / (s_val * 8 + 1);  // s_LM / (s_val + 1/8 byte of bitmap)
  if (o.chunk_width && o.chunk_width > p.dense_numeric) return SPGEMM_ERR_INVALID_ARG;
  p.chunk_width = o.chunk_width ? o.chunk_width : floor_pow2(p.dense_numeric);
  int64_t req = c_cols <= p.chunk_width ? 1 : ceil_div(c_cols, p.chunk_width);
  p.chunks_required = ceil_pow2(req);

  p.group_elems_ms = kMsTile;
  p.group_rows = ceil_div(p.group_elems_ms - 1, p.tau) + 1;
  if (o.chunks_max) {
    p.chunks_max = o.chunks_max;
  } else {
    const int64_t s_ms = kMsSmemBudget, s_histo = 8, s_rowptr = 8, n_sub = 1;
    int64_t num = s_ms - p.group_elems_ms * (s_col + s_val) - s_histo;
    int64_t den = p.group_rows * (n_sub * s_histo + s_rowptr);
    int64_t cm = num > 0 ? num / den : 2;
    p.chunks_max = floor_pow2(cm < 2 ? 2 : cm);
  }
  // the multisplit kernel holds group_rows * chunks bins in shared memory
  while (p.chunks_max > 2 && p.group_rows * p.chunks_max > kMsMaxBins) p.chunks_max /= 2;
  if (p.group_rows * 2 > kMsMaxBins) return SPGEMM_ERR_INVALID_ARG;  // tau far too small

  if (p.chunks_required <= p.chunks_max) {
    p.levels = 1;
    p.v_chunks[0] = p.chunks_required;
  } else {
    const int lr = ilog2_i64(p.chunks_required), lm = ilog2_i64(p.chunks_max);
    p.levels = (lr + lm - 1) / lm;
    if (p.levels > SPGEMM_MAX_LEVELS) return SPGEMM_ERR_INVALID_ARG;
    int64_t prod = 1;
    for (int i = 0; i < p.levels - 1; ++i) {
      p.v_chunks[i] = p.chunks_max;
      prod *= p.chunks_max;
    }
    p.v_chunks[p.levels - 1] = p.chunks_required / prod;
  }
  p.group_elems_op = kOpTile;
  *out = p;
  return SPGEMM_OK;
}

}  // namespace sg

extern "C" int spgemm_plan_params(int64_t c_cols, int64_t s_lm, const spgemm_options* ov,
                                  spgemm_plan* out) {
  return sg::plan_params(c_cols, s_lm, ov, out);
}
