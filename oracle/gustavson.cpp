// CPU oracle for C = A * B on CSR inputs -- TEST INFRASTRUCTURE ONLY.
//
// Only the tests, the smoke check and the benchmark's CPU-baseline leg use this file; the
// library under sparse_gemm_irregular_gb300/ never includes, links or calls it.
//
// What it computes is the plain definition of the product in Gustavson's row-wise form
// (gMAGNUS page, section II-B, Eq. (1) and Algorithm 1): for every row i of A, every
// stored entry A[i,k] (in stored order) scales row k of B, and the scaled entries are
// summed per output column in an ordered map.  The map's keys, in increasing order, are
// row i of C: every column that receives at least one product is kept, even when the
// sum is exactly zero (the structure of C is decided before any value is known, as in
// the symbolic/numeric split of the same section).  Duplicate input entries are separate
// terms.  Next to each sum the oracle keeps the sum of the absolute values of the same
// products, which scales the tests' tolerance.
//
// No blocking, no hashing, no reordering: one std::map per row, single threaded per call.
//
// For the full-size workloads (up to 10^11 products) the same routine is also written with a
// dense accumulator (Gustavson's own: one slot per column of C plus the list of the columns
// touched, sorted at the end of the row).  It visits the products in the same order and adds
// them to each column's sum in the same order as the map, so its sums are bit-identical to
// the map's; only the container differs.  A third routine counts the distinct columns of each
// row (the row sizes of C, i.e. C.row_ptr) with a marker array.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <map>
#include <utility>
#include <vector>

extern "C" {

// Number of intermediate products of each listed row: the sum over the row's entries
// A[i,k] of the length of row k of B.  out[j] is for rows[j].
int oracle_row_ip(const int64_t* a_rp, const int32_t* a_col, const int64_t* b_rp,
                  const int64_t* rows, int64_t nrows, int64_t* out) {
  for (int64_t j = 0; j < nrows; ++j) {
    const int64_t i = rows[j];
    int64_t s = 0;
    for (int64_t p = a_rp[i]; p < a_rp[i + 1]; ++p) {
      const int32_t k = a_col[p];
      s += b_rp[k + 1] - b_rp[k];
    }
    out[j] = s;
  }
  return 0;
}

// Rows rows[0..nrows) of C = A * B.  Output j occupies [out_rp[j], out_rp[j+1]) of
// out_col / out_val / out_abs; out_rp has nrows+1 entries and out_rp[0] = 0.  `cap` is the
// capacity of the three output arrays.  Returns 0, or 1 if the capacity is too small.
int oracle_rows(const int64_t* a_rp, const int32_t* a_col, const double* a_val,
                const int64_t* b_rp, const int32_t* b_col, const double* b_val,
                const int64_t* rows, int64_t nrows, int64_t cap, int64_t* out_rp,
                int32_t* out_col, double* out_val, double* out_abs) {
  int64_t pos = 0;
  out_rp[0] = 0;
  for (int64_t j = 0; j < nrows; ++j) {
    const int64_t i = rows[j];
    std::map<int32_t, std::pair<double, double>> acc;  // column -> (sum, sum of |terms|)
    for (int64_t p = a_rp[i]; p < a_rp[i + 1]; ++p) {
      const int32_t k = a_col[p];
      const double a = a_val[p];
      for (int64_t q = b_rp[k]; q < b_rp[k + 1]; ++q) {
        const double t = a * b_val[q];
        std::pair<double, double>& e = acc[b_col[q]];
        e.first += t;
        e.second += std::fabs(t);
      }
    }
    if (pos + static_cast<int64_t>(acc.size()) > cap) return 1;
    for (const auto& kv : acc) {
      out_col[pos] = kv.first;
      out_val[pos] = kv.second.first;
      out_abs[pos] = kv.second.second;
      ++pos;
    }
    out_rp[j + 1] = pos;
  }
  return 0;
}

// Rows rows[0..nrows) of C = A * B with a dense accumulator over the n columns of C: same
// arguments, outputs and return value as oracle_rows, same sums bit for bit.
int oracle_rows_dense(const int64_t* a_rp, const int32_t* a_col, const double* a_val,
                      const int64_t* b_rp, const int32_t* b_col, const double* b_val, int64_t n,
                      const int64_t* rows, int64_t nrows, int64_t cap, int64_t* out_rp,
                      int32_t* out_col, double* out_val, double* out_abs) {
  std::vector<double> sum(static_cast<size_t>(n), 0.0), abs_sum(static_cast<size_t>(n), 0.0);
  std::vector<char> seen(static_cast<size_t>(n), 0);
  std::vector<int32_t> touched;
  int64_t pos = 0;
  out_rp[0] = 0;
  for (int64_t j = 0; j < nrows; ++j) {
    const int64_t i = rows[j];
    touched.clear();
    for (int64_t p = a_rp[i]; p < a_rp[i + 1]; ++p) {
      const int32_t k = a_col[p];
      const double a = a_val[p];
      for (int64_t q = b_rp[k]; q < b_rp[k + 1]; ++q) {
        const int32_t c = b_col[q];
        const double t = a * b_val[q];
        if (!seen[c]) {
          seen[c] = 1;
          touched.push_back(c);
        }
        sum[c] += t;
        abs_sum[c] += std::fabs(t);
      }
    }
    if (pos + static_cast<int64_t>(touched.size()) > cap) return 1;
    std::sort(touched.begin(), touched.end());
    for (const int32_t c : touched) {
      out_col[pos] = c;
      out_val[pos] = sum[c];
      out_abs[pos] = abs_sum[c];
      ++pos;
      sum[c] = 0.0;
      abs_sum[c] = 0.0;
      seen[c] = 0;
    }
    out_rp[j + 1] = pos;
  }
  return 0;
}

// Number of distinct columns of each listed row of C = A * B (every column receiving at least
// one product counts, whatever its sum).  out[j] is for rows[j].
int oracle_row_nnz(const int64_t* a_rp, const int32_t* a_col, const int64_t* b_rp, const int32_t* b_col,
                   int64_t n, const int64_t* rows, int64_t nrows, int64_t* out) {
  std::vector<int64_t> mark(static_cast<size_t>(n), -1);
  for (int64_t j = 0; j < nrows; ++j) {
    const int64_t i = rows[j];
    int64_t cnt = 0;
    for (int64_t p = a_rp[i]; p < a_rp[i + 1]; ++p) {
      const int32_t k = a_col[p];
      for (int64_t q = b_rp[k]; q < b_rp[k + 1]; ++q) {
        const int32_t c = b_col[q];
        if (mark[c] != j) {
          mark[c] = j;
          ++cnt;
        }
      }
    }
    out[j] = cnt;
  }
  return 0;
}

}  // extern "C"
