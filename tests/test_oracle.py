"""Pins for the CPU oracle: each test checks it against something other than itself.

Brute force on small dense matrices, exact closed forms (identity, permutations, banded
squares, disjoint structure), integer-valued sums that must be exact in any order, and
the structural rule that a column receiving products whose sum is exactly 0 stays in C
(gMAGNUS page, section II-B: the symbolic phase fixes the row sizes before any value).
"""
import numpy as np
import pytest

import oracle
import synth
from synth import CSR


@pytest.fixture(params=["map", "dense"])
def acc(request):
    """Both accumulators of the oracle run through every pin."""
    return request.param


def dense(m: CSR, absolute=False, pattern=False):
    d = np.zeros((m.rows, m.cols))
    rows = np.repeat(np.arange(m.rows), np.diff(m.row_ptr))
    v = np.ones(m.nnz) if pattern else (np.abs(m.val) if absolute else m.val)
    np.add.at(d, (rows, m.col), v)
    return d


def to_dense_out(c: CSR):
    d = np.zeros((c.rows, c.cols))
    present = np.zeros((c.rows, c.cols), dtype=bool)
    rows = np.repeat(np.arange(c.rows), np.diff(c.row_ptr))
    d[rows, c.col] = c.val
    present[rows, c.col] = True
    return d, present


def assert_sorted_rows(c: CSR):
    for i in range(c.rows):
        cols, _ = c.row(i)
        assert np.all(np.diff(cols) > 0), f"row {i} not strictly increasing"


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("dup,empty,sort", [(False, False, True), (True, True, False),
                                             (True, False, True), (False, True, False)])
def test_bruteforce_dense(seed, dup, empty, sort, acc):
    m, k, n = 23 + seed, 31, 17 + 2 * seed          # rectangular: catches a transposed operand
    A = synth.random_sparse(m, k, 0.15, seed, duplicates=dup, empty_rows=empty, sort_rows=sort)
    B = synth.random_sparse(k, n, 0.2, seed + 100, duplicates=dup, empty_rows=empty, sort_rows=sort)
    C, ab = oracle.spgemm(A, B, accumulator=acc)
    C.check()
    assert_sorted_rows(C)
    ref = dense(A) @ dense(B)
    ref_abs = dense(A, absolute=True) @ dense(B, absolute=True)
    struct = (dense(A, pattern=True) @ dense(B, pattern=True)) > 0
    got, present = to_dense_out(C)
    assert np.array_equal(present, struct)
    assert np.all(np.abs(got - ref) <= 1e-14 * ref_abs + 1e-300)
    # the abs-sum output equals |A| |B| entrywise (same terms, nonnegative)
    abs_d = np.zeros_like(got)
    rows = np.repeat(np.arange(C.rows), np.diff(C.row_ptr))
    abs_d[rows, C.col] = ab
    assert np.all(np.abs(abs_d - ref_abs) <= 1e-14 * ref_abs)


def test_integer_values_exact(acc):
    A = synth.random_sparse(60, 50, 0.2, 7, duplicates=True, integer_values=True, sort_rows=False)
    B = synth.random_sparse(50, 70, 0.2, 8, duplicates=True, integer_values=True, sort_rows=False)
    C, _ = oracle.spgemm(A, B, accumulator=acc)
    got, present = to_dense_out(C)
    ref = dense(A) @ dense(B)
    assert np.array_equal(got, ref)  # every partial sum is a small integer: exact
    assert np.array_equal(present, (dense(A, pattern=True) @ dense(B, pattern=True)) > 0)


def identity(n):
    return CSR(n, n, np.arange(n + 1, dtype=np.int64), np.arange(n, dtype=np.int32), np.ones(n))


def perm_matrix(perm, scale=None):
    n = len(perm)
    v = np.ones(n) if scale is None else scale
    return CSR(n, n, np.arange(n + 1, dtype=np.int64), perm.astype(np.int32), v.astype(np.float64))


def test_identity(acc):
    A = synth.random_sparse(40, 40, 0.1, 3)
    for C, _ in (oracle.spgemm(A, identity(40), accumulator=acc), oracle.spgemm(identity(40), A, accumulator=acc)):
        assert np.array_equal(C.row_ptr, A.row_ptr)
        assert np.array_equal(C.col, A.col)
        assert np.array_equal(C.val, A.val)  # single term times 1.0: bit-exact


def test_permutations(acc):
    n = 50
    A = synth.random_sparse(n, n, 0.1, 4)
    perm = (synth.draws(0, 9, 0, n) % np.uint64(1 << 62)).argsort()
    P = perm_matrix(perm)                 # P[i, perm[i]] = 1
    C, _ = oracle.spgemm(P, A, accumulator=acc)            # row i of C is row perm[i] of A
    for i in range(n):
        c1, v1 = C.row(i)
        c2, v2 = A.row(int(perm[i]))
        assert np.array_equal(c1, c2) and np.array_equal(v1, v2)
    C2, _ = oracle.spgemm(A, P, accumulator=acc)           # column j of A moves to column perm[j]
    for i in range(n):
        cols, vals = A.row(i)
        new = perm[cols]
        order = np.argsort(new)
        c1, v1 = C2.row(i)
        assert np.array_equal(c1, new[order]) and np.array_equal(v1, vals[order])


@pytest.mark.parametrize("n,h", [(50, 1), (64, 3), (200, 3), (97, 5)])
def test_banded_square(n, h, acc):
    A = synth.banded(n, h)
    A.val = np.ones(A.nnz)
    C, _ = oracle.spgemm(A, A, accumulator=acc)
    assert C.nnz == (4 * h + 1) * n - 2 * h * (2 * h + 1)
    for i in range(2 * h, n - 2 * h):     # interior rows: exact triangle profile
        cols, vals = C.row(i)
        assert np.array_equal(cols, np.arange(i - 2 * h, i + 2 * h + 1))
        assert np.array_equal(vals, (2 * h + 1) - np.abs(cols - i).astype(float))


def test_disjoint_structure(acc):
    n = 64
    B = synth.random_sparse(n, 90, 0.1, 5)
    perm = (synth.draws(1, 9, 0, n) % np.uint64(1 << 62)).argsort()
    scale = synth.uniform(0, 11, 0, n, 0.5, 2.0)
    P = perm_matrix(perm, scale)
    C, _ = oracle.spgemm(P, B, accumulator=acc)
    for i in range(n):
        cols, vals = C.row(i)
        bc, bv = B.row(int(perm[i]))
        assert len(cols) == len(bc)       # nnz of the row equals its intermediate products
        order = np.argsort(bc)
        assert np.array_equal(cols, bc[order])
        assert np.array_equal(vals, scale[i] * bv[order])  # one product per entry: exact


def test_cancellation_kept(acc):
    A = CSR(1, 2, np.array([0, 2], np.int64), np.array([0, 1], np.int32), np.array([1.0, 1.0]))
    B = CSR(2, 1, np.array([0, 1, 2], np.int64), np.array([0, 0], np.int32), np.array([2.0, -2.0]))
    C, ab = oracle.spgemm(A, B, accumulator=acc)
    assert C.nnz == 1 and C.val[0] == 0.0 and ab[0] == 4.0


def test_empty_and_degenerate(acc):
    Z = CSR(5, 7, np.zeros(6, np.int64), np.zeros(0, np.int32), np.zeros(0))
    B = synth.random_sparse(7, 4, 0.5, 1)
    C, _ = oracle.spgemm(Z, B, accumulator=acc)
    assert C.nnz == 0 and C.rows == 5 and C.cols == 4
    E = CSR(0, 7, np.zeros(1, np.int64), np.zeros(0, np.int32), np.zeros(0))
    C, _ = oracle.spgemm(E, B, accumulator=acc)
    assert C.rows == 0 and C.nnz == 0


def test_threaded_rows_match_single():
    A = synth.random_sparse(300, 200, 0.05, 12)
    B = synth.random_sparse(200, 250, 0.05, 13)
    r1 = oracle.spgemm_rows(A, B, np.arange(300), threads=1)
    r4 = oracle.spgemm_rows(A, B, np.arange(300), threads=4)
    for x, y in zip(r1, r4):
        assert np.array_equal(x, y)


def test_row_ip_definition():
    A = synth.random_sparse(30, 20, 0.2, 2, duplicates=True)
    B = synth.random_sparse(20, 25, 0.2, 3, duplicates=True)
    ip = oracle.row_ip(A, B)
    ref = (dense(A, pattern=True) @ dense(B, pattern=True)).sum(axis=1)
    assert np.array_equal(ip, ref.astype(np.int64))


@pytest.mark.parametrize("case", ["rmat", "random_dup_unsorted", "uniform8", "band"])
def test_dense_accumulator_bit_identical_to_map(case):
    """The dense accumulator visits the products in the map's order and adds them to each
    column's sum in the same order, so every output array is identical bit for bit."""
    if case == "rmat":
        A = B = synth.rmat(12, 16, seed=2)
    elif case == "random_dup_unsorted":
        A = synth.random_sparse(400, 300, 0.03, 5, duplicates=True, empty_rows=True, sort_rows=False)
        B = synth.random_sparse(300, 700, 0.02, 6, duplicates=True, empty_rows=True, sort_rows=False)
    elif case == "uniform8":
        A = B = synth.uniform_rows(2048, 8, seed=1)
    else:
        A = B = synth.banded(5000, 3, seed=3)
    rows = np.arange(A.rows)
    m = oracle.spgemm_rows(A, B, rows, threads=4)
    d = oracle.spgemm_rows(A, B, rows, threads=4, accumulator="dense")
    for x, y in zip(m, d):
        assert x.dtype == y.dtype and np.array_equal(x, y)


@pytest.mark.parametrize("seed", range(4))
def test_row_nnz_definition(seed):
    """Row sizes of C: the number of columns reached by the pattern product (brute force),
    with duplicates and unsorted rows; equal to the map oracle's row sizes."""
    A = synth.random_sparse(40, 35, 0.15, seed, duplicates=True, empty_rows=True, sort_rows=False)
    B = synth.random_sparse(35, 60, 0.2, seed + 20, duplicates=True, empty_rows=True, sort_rows=False)
    ref = ((dense(A, pattern=True) @ dense(B, pattern=True)) > 0).sum(axis=1)
    assert np.array_equal(oracle.row_nnz(A, B), ref.astype(np.int64))
    rows = np.arange(A.rows)[::-1].copy()  # any row order
    assert np.array_equal(oracle.row_nnz(A, B, rows, threads=3), ref[::-1].astype(np.int64))
    C, _ = oracle.spgemm(A, B)
    assert np.array_equal(oracle.row_nnz(A, B), np.diff(C.row_ptr))


def test_row_nnz_banded_closed_form():
    A = synth.banded(10_000, 3)
    nnz = oracle.row_nnz(A, A, threads=4)
    assert nnz.sum() == 13 * A.rows - 42
    assert np.all(nnz[6:-6] == 13)
