"""Seeded synthetic sparse-matrix generators shared by the oracle tests and the GPU path.

This module only builds inputs: it holds none of the SpGEMM arithmetic (no products, no
accumulation, no row sizes of C).  Every random number comes from one counter-based
generator, splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014), evaluated at ``key(seed, stream) + (index + 1) * gamma``, so a
draw depends only on (seed, stream, index) and generation is reproducible on any host.

Workloads (stand-ins for the pages' PaRMAT R-MAT pairs and the Markov-clustering
expansion; the SuiteSparse matrices are not reproduced):

* ``uniform_rows``  -- exactly ``per_row`` distinct uniform columns per row (Floyd's
  sampling), values U[-1, 1).
* ``banded``        -- columns i-h .. i+h clipped at the edges, values U[-1, 1).
* ``rmat``          -- R-MAT edges with quadrant probabilities (a, b, c, d), one uniform draw
  per recursion level, no noise and no vertex permutation, duplicates merged, self loops
  kept, values U[0, 1) drawn after merging in CSR order (gMAGNUS page, section IV-A,
  Graph500 parameters a = 0.57, b = c = 0.19).
* ``mcl_matrix``    -- R-MAT pattern plus the identity, every column scaled to sum 1
  (Trident page, Markov clustering experiment: expansion step M*M).
"""
from __future__ import annotations

from dataclasses import dataclass

import concurrent.futures
import os

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream ids: one per independent use
STREAM_STRUCT = 1
STREAM_VALUES = 2
STREAM_SAMPLE = 3


def _fin(z: np.ndarray) -> np.ndarray:
    """splitmix64 output function (in place on a uint64 array)."""
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        z = np.array([(seed * 0x9E3779B97F4A7C15 + stream * 0xD1B54A32D192ED03 + 1)
                      & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return _fin(z)[0]


def draws(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """uint64 draws number start .. start+count-1 of (seed, stream)."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z = idx * _GAMMA
        z += _key(seed, stream)
        return _fin(z)


def to_unit(d: np.ndarray) -> np.ndarray:
    """Top 53 bits of each draw as a double in [0, 1)."""
    return (d >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def uniform(seed: int, stream: int, start: int, count: int, lo: float, hi: float) -> np.ndarray:
    u = to_unit(draws(seed, stream, start, count))
    return lo + (hi - lo) * u


@dataclass
class CSR:
    """Host CSR matrix: int64 row_ptr (rows+1), int32 col (nnz), float64 val (nnz)."""
    rows: int
    cols: int
    row_ptr: np.ndarray
    col: np.ndarray
    val: np.ndarray

    @property
    def nnz(self) -> int:
        return int(self.row_ptr[-1])

    def row(self, i: int):
        a, b = int(self.row_ptr[i]), int(self.row_ptr[i + 1])
        return self.col[a:b], self.val[a:b]

    def check(self) -> None:
        assert self.row_ptr.dtype == np.int64 and self.col.dtype == np.int32
        assert self.val.dtype == np.float64
        assert self.row_ptr.shape == (self.rows + 1,) and self.row_ptr[0] == 0
        assert np.all(np.diff(self.row_ptr) >= 0)
        assert self.col.shape == (self.nnz,) and self.val.shape == (self.nnz,)
        if self.nnz:
            assert self.col.min() >= 0 and self.col.max() < self.cols

    def bytes(self) -> int:
        return (self.rows + 1) * 8 + self.nnz * 12


def csr_from_coo(rows: int, cols: int, r: np.ndarray, c: np.ndarray, v: np.ndarray,
                 merge: bool = False) -> CSR:
    """Build CSR ordered by (row, col).  With ``merge`` duplicate (row, col) pairs are
    collapsed into one entry keeping the first value (patterns only; values are drawn
    after merging by the callers)."""
    key = r.astype(np.int64) * np.int64(cols) + c.astype(np.int64)
    if merge:
        key, first = np.unique(key, return_index=True)
        v = v[first]
    else:
        order = np.argsort(key, kind="stable")
        key, v = key[order], v[order]
    rr = key // cols
    cc = (key % cols).astype(np.int32)
    counts = np.bincount(rr, minlength=rows).astype(np.int64)
    rp = np.zeros(rows + 1, dtype=np.int64)
    np.cumsum(counts, out=rp[1:])
    return CSR(rows, cols, rp, cc, np.ascontiguousarray(v, dtype=np.float64))


def transpose(m: CSR) -> CSR:
    """The transpose as CSR (input preparation for products such as A * A^T)."""
    r = np.repeat(np.arange(m.rows, dtype=np.int64), np.diff(m.row_ptr))
    return csr_from_coo(m.cols, m.rows, m.col.astype(np.int64), r.astype(np.int32), m.val)


def aggregation(n: int, coarse: int, seed: int = 0, per_row: int = 1) -> CSR:
    """n x coarse restriction-style operator: row i has ``per_row`` distinct columns drawn from
    [0, coarse), values 1 / per_row (a tall, skinny B for rectangular products A * R)."""
    cols = np.empty((n, per_row), dtype=np.int64)
    for j in range(per_row):
        cols[:, j] = (draws(seed, 11 + j, 0, n) % np.uint64(coarse)).astype(np.int64)
    r = np.repeat(np.arange(n, dtype=np.int64), per_row)
    c = cols.reshape(-1)
    m = csr_from_coo(n, coarse, r, c.astype(np.int32), np.full(n * per_row, 1.0 / per_row), merge=True)
    return m


def uniform_rows(n: int, per_row: int, seed: int = 0, lo: float = -1.0, hi: float = 1.0) -> CSR:
    """n x n, exactly ``per_row`` distinct columns per row chosen uniformly by Floyd's
    algorithm, columns stored sorted, values U[lo, hi)."""
    assert per_row <= n
    cols = np.empty((n, per_row), dtype=np.int64)
    for t, j in enumerate(range(n - per_row, n)):
        d = draws(seed, STREAM_STRUCT, t * n, n)
        pick = (d % np.uint64(j + 1)).astype(np.int64)
        taken = (cols[:, :t] == pick[:, None]).any(axis=1) if t else np.zeros(n, bool)
        cols[:, t] = np.where(taken, j, pick)
    cols.sort(axis=1)
    rp = np.arange(0, n * per_row + 1, per_row, dtype=np.int64)
    val = uniform(seed, STREAM_VALUES, 0, n * per_row, lo, hi)
    return CSR(n, n, rp, cols.reshape(-1).astype(np.int32), val)


def banded(n: int, half_width: int, seed: int = 0, lo: float = -1.0, hi: float = 1.0) -> CSR:
    """n x n band: row i holds columns max(0, i-h) .. min(n-1, i+h); values U[lo, hi)."""
    i = np.arange(n, dtype=np.int64)
    lo_c = np.maximum(0, i - half_width)
    hi_c = np.minimum(n - 1, i + half_width)
    counts = hi_c - lo_c + 1
    rp = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(counts, out=rp[1:])
    nnz = int(rp[-1])
    row_of = np.repeat(i, counts)
    col = (lo_c[row_of] + (np.arange(nnz, dtype=np.int64) - rp[row_of])).astype(np.int32)
    val = uniform(seed, STREAM_VALUES, 0, nnz, lo, hi)
    return CSR(n, n, rp, col, val)


def rmat_edges(scale: int, n_edges: int, a: float, b: float, c: float, seed: int = 0,
               block: int = 1 << 22):
    """R-MAT edge list: for every edge and every level (most significant bit first) one
    uniform draw u picks quadrant (0,0) if u < a, (0,1) if u < a+b, (1,0) if u < a+b+c,
    else (1,1).  Blocks of edges are independent (counter-based draws), so they are generated
    by a thread pool (numpy releases the GIL on these array operations); the result does not
    depend on the number of threads."""
    rows = np.empty(n_edges, dtype=np.int64)
    cols = np.empty(n_edges, dtype=np.int64)
    ab, abc = a + b, a + b + c
    key = _key(seed, STREAM_STRUCT)

    def one(e0):
        e1 = min(n_edges, e0 + block)
        ne = e1 - e0
        r = np.zeros(ne, dtype=np.int64)
        cc = np.zeros(ne, dtype=np.int64)
        with np.errstate(over="ignore"):
            base = np.arange(e0, e1, dtype=np.uint64) * np.uint64(scale)
            for lvl in range(scale):
                # draw index = edge * scale + level
                u = to_unit(_fin((base + np.uint64(lvl + 1)) * _GAMMA + key))
                rbit = (u >= ab).astype(np.int64)
                cbit = (((u >= a) & (u < ab)) | (u >= abc)).astype(np.int64)
                r = (r << 1) | rbit
                cc = (cc << 1) | cbit
        rows[e0:e1] = r
        cols[e0:e1] = cc

    starts = list(range(0, n_edges, block))
    workers = max(1, min(len(starts), os.cpu_count() or 1, 16))
    if workers == 1:
        for e0 in starts:
            one(e0)
    else:
        with concurrent.futures.ThreadPoolExecutor(workers) as ex:
            list(ex.map(one, starts))
    return rows, cols


def rmat(scale: int, edge_factor: int, a: float = 0.57, b: float = 0.19, c: float = 0.19,
         seed: int = 0, lo: float = 0.0, hi: float = 1.0) -> CSR:
    """2^scale square R-MAT matrix, edge_factor * 2^scale draws, duplicates merged,
    values U[lo, hi) in CSR order after merging."""
    n = 1 << scale
    with np.errstate(over="ignore"):
        r, cc = rmat_edges(scale, edge_factor * n, a, b, c, seed)
    m = csr_from_coo(n, n, r, cc, np.zeros(len(r)), merge=True)
    m.val = uniform(seed, STREAM_VALUES, 0, m.nnz, lo, hi)
    return m


def mcl_matrix(scale: int, edge_factor: int, seed: int = 0) -> CSR:
    """Markov-clustering input: merged R-MAT pattern plus self loops, every stored value 1
    before scaling, then M[i, j] = 1 / (number of entries in column j)."""
    n = 1 << scale
    with np.errstate(over="ignore"):
        r, cc = rmat_edges(scale, edge_factor * n, 0.57, 0.19, 0.19, seed)
    d = np.arange(n, dtype=np.int64)
    m = csr_from_coo(n, n, np.concatenate([r, d]), np.concatenate([cc, d]),
                     np.zeros(len(r) + n), merge=True)
    colcount = np.bincount(m.col, minlength=n).astype(np.float64)
    m.val = 1.0 / colcount[m.col]
    return m


def random_sparse(m: int, n: int, density: float, seed: int, duplicates: bool = False,
                  empty_rows: bool = False, lo: float = -1.0, hi: float = 1.0,
                  integer_values: bool = False, sort_rows: bool = True) -> CSR:
    """Small random CSR for pins and edge cases.  With ``duplicates`` a row may hold the
    same column more than once; with ``empty_rows`` about a quarter of the rows are
    empty; ``sort_rows=False`` shuffles the entries inside each row."""
    total = int(round(m * n * density))
    d = draws(seed, STREAM_STRUCT, 0, 2 * total + m)
    r = (d[:total] % np.uint64(m)).astype(np.int64)
    c = (d[total:2 * total] % np.uint64(n)).astype(np.int64)
    if empty_rows:
        keep_row = (d[2 * total:] % np.uint64(4)) != 0
        sel = keep_row[r]
        r, c = r[sel], c[sel]
    mat = csr_from_coo(m, n, r, c, np.zeros(len(r)), merge=not duplicates)
    if integer_values:
        mat.val = (draws(seed, STREAM_VALUES, 0, mat.nnz) % np.uint64(7)).astype(np.float64) - 3.0
    else:
        mat.val = uniform(seed, STREAM_VALUES, 0, mat.nnz, lo, hi)
    if not sort_rows:
        key = draws(seed, STREAM_SAMPLE, 0, mat.nnz)
        order = np.lexsort((key, np.repeat(np.arange(m), np.diff(mat.row_ptr))))
        mat.col, mat.val = mat.col[order], mat.val[order]
    return mat


def with_values(m: CSR, values: np.ndarray) -> CSR:
    return CSR(m.rows, m.cols, m.row_ptr, m.col, np.ascontiguousarray(values, np.float64))


# The five workloads.  (id, name, description, builder)
CONFIGS = {
    1: ("uniform8_n2048", "C=A*A, A 2048x2048, 8 distinct uniform columns per row, U[-1,1)",
        lambda seed=0: uniform_rows(2048, 8, seed)),
    2: ("band7_n1e6", "C=A*A, A 1,000,000^2 band (cols i-3..i+3), U[-1,1)",
        lambda seed=0: banded(1_000_000, 3, seed)),
    3: ("rmat_s18_ef16", "C=A*A, R-MAT scale 18, edge factor 16, (0.57,0.19,0.19,0.05), U[0,1)",
        lambda seed=0: rmat(18, 16, seed=seed)),
    4: ("rmat_s21_ef32", "C=A*A, R-MAT scale 21, edge factor 32, (0.57,0.19,0.19,0.05), U[0,1)",
        lambda seed=0: rmat(21, 32, seed=seed)),
    5: ("mcl_rmat_s20_ef16", "C=M*M, M = column-stochastic (R-MAT scale 20, edge factor 16, + I)",
        lambda seed=0: mcl_matrix(20, 16, seed)),
}


def config(cid: int, seed: int = 0) -> CSR:
    return CONFIGS[cid][2](seed)
