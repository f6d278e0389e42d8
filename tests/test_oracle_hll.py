"""Pins for the oracle's HyperLogLog row-size estimates (Ocean page: HyperLogLog background,
construct-and-merge scheme of Figure 3, overflow evaluation).  Each test checks the oracle
against something other than its own formulas: a bit-string reading of the register index and
rank, the sketch of the exact column set of C's rows (from the Gustavson oracle), closed forms
of the estimator, and known cardinalities within the estimator's stated error."""
import math

import numpy as np
import pytest

import oracle
import synth
from oracle import hll


@pytest.mark.parametrize("m", [32, 64])
def test_index_and_rank_bitstrings(m):
    rng = np.random.default_rng(5)
    cols = rng.integers(0, 2**31 - 1, 2000)
    cols[:3] = [0, 1, 2**31 - 2]
    idx, rank = hll.index_rank(cols, m)
    b = int(math.log2(m))
    for c, i, r, h in zip(cols, idx, rank, hll.mix32(cols)):
        bits = format(int(h), "032b")
        assert int(bits[32 - b:], 2) == i
        rest = bits[:32 - b]
        expect = rest.index("1") + 1 if "1" in rest else 33 - b
        assert r == expect


def test_mix32_is_a_bijection_on_a_range():
    h = hll.mix32(np.arange(1 << 20))
    assert len(np.unique(h)) == 1 << 20
    assert int(hll.mix32(np.array([0]))[0]) == 0  # every step of the finaliser fixes zero


@pytest.mark.parametrize("m", [32, 64])
@pytest.mark.parametrize("seed", [0, 1])
def test_merged_sketch_is_the_sketch_of_the_row_of_c(m, seed):
    """HyperLogLog depends only on the set of distinct columns, so the merge of the B-row
    sketches must equal the sketch of the columns of C's row, taken from the exact product."""
    A = synth.random_sparse(120, 90, 0.08, seed, duplicates=True, empty_rows=True, sort_rows=False)
    B = synth.random_sparse(90, 3000, 0.02, seed + 7, duplicates=True, empty_rows=True)
    merged = hll.merge_rows(A, hll.sketch_rows(B, m))
    C, _ = oracle.spgemm(A, B)
    for i in range(A.rows):
        cols, _ = C.row(i)
        assert np.array_equal(merged[i], hll.sketch(cols, m)), i


@pytest.mark.parametrize("m", [32, 64])
def test_estimator_closed_forms(m):
    assert hll.estimate(np.zeros(m, np.uint8)) == 0.0
    one = hll.sketch(np.array([12345]), m)
    assert (one > 0).sum() == 1
    assert hll.estimate(one) == pytest.approx(m * math.log(m / (m - 1)), rel=0, abs=0)


@pytest.mark.parametrize("m", [32, 64])
@pytest.mark.parametrize("n", [3000, 30000, 300000])
def test_estimator_error_within_its_bound(m, n):
    """Relative error 1.04/sqrt(m) (the page's figure): four standard errors on seeded sets."""
    rng = np.random.default_rng(n + m)
    cols = rng.choice(2**31 - 1, size=n, replace=False)
    e = hll.estimate(hll.sketch(cols, m))
    assert abs(e / n - 1) <= 4 * 1.04 / math.sqrt(m)


def test_capacities_bound_and_overflow_rate():
    A = synth.rmat(11, 8, seed=3)
    ip = oracle.row_ip(A, A)
    C, _ = oracle.spgemm(A, A, threads=8)
    nnz = np.diff(C.row_ptr)
    for m in (32, 64):
        cap = hll.capacities(A, A, m, hll.coefficient(m), ip)
        assert np.all(cap <= ip) and np.all((cap > 0) == (ip > 0))
        over = (nnz > cap).sum() / max((ip > 0).sum(), 1)
        assert over < 0.05, (m, over)


def test_registers_and_coefficient_rules():
    assert hll.registers_for(47 * 100, 100) == 32 and hll.registers_for(48 * 100, 100) == 64
    assert hll.coefficient(32) == 2.0 and hll.coefficient(64) == 1.5


def _alpha_from_integral(m):
    """alpha_m of HyperLogLog from its defining integral (Flajolet, Fusy, Gandouet, Meunier 2007,
    the reference the Ocean page gives for the estimator's bias correction):
    alpha_m = 1 / (m * integral_0^inf (log2((2 + u) / (1 + u)))^m du)."""
    integrate = pytest.importorskip("scipy.integrate")
    v, _ = integrate.quad(lambda u: math.log2((2.0 + u) / (1.0 + u)) ** m, 0.0, math.inf, limit=500)
    return 1.0 / (m * v)


@pytest.mark.parametrize("m", [16, 32, 64])
def test_estimator_constant_against_its_integral(m):
    """The raw estimator alpha_m m^2 / sum 2^-M, read through estimate() on sketches where linear
    counting does not apply (no empty register), against alpha_m integrated numerically.  The
    constants are printed to three decimals, so they agree to 5e-4; a swapped alpha_32 / alpha_64
    (1.7% apart) or alpha_16's 0.673 at m = 64 lies far outside."""
    alpha = _alpha_from_integral(m)
    for level in (6, 11, 17):
        regs = np.full(m, level, dtype=np.uint8)
        regs[::3] = level + 1
        z = sum(2.0 ** (-int(r)) for r in regs)
        assert abs(hll.estimate(regs) * z / (m * m) - alpha) <= 5e-4


@pytest.mark.parametrize("m,n", [(32, 640), (64, 1280)])
def test_estimator_unbiased_on_average(m, n):
    """Mean of estimate / cardinality over 2000 seeded sets of about 20m distinct columns: the
    estimator is unbiased in this range, and the mean's standard error is below 0.5%, so it lies
    within 1% of 1.  A wrong alpha_m shifts every estimate by the same factor and fails this."""
    rng = np.random.default_rng(1000 + m + n)
    ratios = []
    for _ in range(2000):
        cols = np.unique(rng.integers(0, 2**31 - 1, size=n))
        ratios.append(hll.estimate(hll.sketch(cols, m)) / len(cols))
    assert abs(float(np.mean(ratios)) - 1.0) <= 0.01


def test_capacities_worked_rows():
    """Capacities worked by hand on tiny products (two columns land in distinct registers; the
    estimate then comes from linear counting, m ln(m / V) with V empty registers):
      row 0: one product, column c0          -> IP 1, estimate m ln(m/(m-1)); capped at IP = 1
      row 1: two products on column c0        -> IP 2, ceil(coef * m ln(m/(m-1)))
      row 2: two products on columns c0, c1   -> IP 2, capped at 2
      row 3: four products on columns c0, c1  -> IP 4, ceil(coef * m ln(m/(m-2)))
      row 4: no product                       -> 0
    m = 64, coef 1.5: rows 1 and 3 give ceil(1.5119) = 2 and ceil(3.0477) = 4 (floor or
    rounding would give 1 and 3); m = 32, coef 2.0: ceil(2.0319) = 3 and ceil(4.0954) = 5."""
    from synth import CSR
    c0 = 5
    c1 = next(c for c in range(6, 10000) if hll.index_rank(np.array([c]), 64)[0][0]
              != hll.index_rank(np.array([c0]), 64)[0][0]
              and hll.index_rank(np.array([c]), 32)[0][0] != hll.index_rank(np.array([c0]), 32)[0][0])
    # B: row 0 = {c0}, row 1 = {c1}; A selects them
    B = CSR(2, 10000, np.array([0, 1, 2], np.int64), np.array([c0, c1], np.int32), np.ones(2))
    A = CSR(5, 2, np.array([0, 1, 3, 5, 9, 9], np.int64), np.array([0, 0, 0, 0, 1, 0, 1, 0, 1], np.int32),
            np.ones(9))
    ip = oracle.row_ip(A, B)
    assert list(ip) == [1, 2, 2, 4, 0]
    for m, coef, expect in ((64, 1.5, [1, 2, 2, 4, 0]), (32, 2.0, [1, 2, 2, 4, 0])):
        cap = hll.capacities(A, B, m, coef, ip)
        assert list(cap) == expect
    # the same rows with IP large enough that the estimate, not IP, decides
    A2 = CSR(2, 2, np.array([0, 3, 9], np.int64), np.array([0, 0, 0, 0, 1, 0, 1, 0, 1], np.int32), np.ones(9))
    ip2 = oracle.row_ip(A2, B)
    assert list(ip2) == [3, 6]
    assert list(hll.capacities(A2, B, 64, 1.5, ip2)) == [2, 4]
    assert list(hll.capacities(A2, B, 32, 2.0, ip2)) == [3, 5]
    # the closed forms behind them
    assert math.ceil(1.5 * 64 * math.log(64 / 63)) == 2 and math.ceil(1.5 * 64 * math.log(64 / 62)) == 4
    assert math.ceil(2.0 * 32 * math.log(32 / 31)) == 3 and math.ceil(2.0 * 32 * math.log(32 / 30)) == 5
