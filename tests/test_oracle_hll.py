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
