"""CPU oracle for C = A * B (TEST INFRASTRUCTURE ONLY).

Used by tests/, the smoke check and the benchmark's CPU-baseline leg; the library never
imports it.  The arithmetic lives in gustavson.cpp: a single-threaded Gustavson product
with an ordered-map accumulator per row (gMAGNUS page, section II-B, Eq. (1),
Algorithm 1).  ``spgemm_rows`` may split a row list across host threads; every thread
runs the same unchanged per-row routine on its own rows.

The dense-accumulator routine (``accumulator="dense"``) and the row-size counter
(``row_nnz``) serve the full-size comparisons; the dense routine adds the same products in the
same order as the map, so both give the same bits.

Parity status: pinned (tests/test_oracle.py) against dense brute force on small inputs,
closed forms (A*I = A, permutations, banded squares, disjoint structure), integer-valued
exact sums and the printed chunk tables do not apply here (they pin the planner).  Both
accumulators and the row-size counter run through the same pins, and the dense accumulator is
checked bit for bit against the map on R-MAT and random inputs.
"""
from __future__ import annotations

import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.oracle_row_ip.argtypes = [p, p, p, p, i64, p]
        lib.oracle_row_ip.restype = ctypes.c_int
        lib.oracle_rows.argtypes = [p, p, p, p, p, p, p, i64, i64, p, p, p, p]
        lib.oracle_rows.restype = ctypes.c_int
        lib.oracle_rows_dense.argtypes = [p, p, p, p, p, p, i64, p, i64, i64, p, p, p, p]
        lib.oracle_rows_dense.restype = ctypes.c_int
        lib.oracle_row_nnz.argtypes = [p, p, p, p, i64, p, i64, p]
        lib.oracle_row_nnz.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def row_ip(A, B, rows=None) -> np.ndarray:
    """Intermediate products per row of A*B (all rows, or the listed ones)."""
    lib = _load()
    rows = np.arange(A.rows, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    out = np.zeros(len(rows), dtype=np.int64)
    lib.oracle_row_ip(_ptr(A.row_ptr), _ptr(A.col), _ptr(B.row_ptr), _ptr(rows), len(rows), _ptr(out))
    return out


def _rows_one(A, B, rows: np.ndarray, accumulator: str = "map"):
    lib = _load()
    if accumulator == "map":
        cap = int(row_ip(A, B, rows).sum())
    else:  # the exact sizes are cheap next to the products, and keep the outputs small
        cap = int(row_nnz(A, B, rows).sum())
    rp = np.zeros(len(rows) + 1, dtype=np.int64)
    col = np.zeros(max(cap, 1), dtype=np.int32)
    val = np.zeros(max(cap, 1), dtype=np.float64)
    ab = np.zeros(max(cap, 1), dtype=np.float64)
    if accumulator == "map":
        rc = lib.oracle_rows(_ptr(A.row_ptr), _ptr(A.col), _ptr(A.val), _ptr(B.row_ptr), _ptr(B.col),
                             _ptr(B.val), _ptr(rows), len(rows), cap, _ptr(rp), _ptr(col), _ptr(val),
                             _ptr(ab))
    elif accumulator == "dense":
        rc = lib.oracle_rows_dense(_ptr(A.row_ptr), _ptr(A.col), _ptr(A.val), _ptr(B.row_ptr), _ptr(B.col),
                                   _ptr(B.val), B.cols, _ptr(rows), len(rows), cap, _ptr(rp), _ptr(col),
                                   _ptr(val), _ptr(ab))
    else:
        raise ValueError(accumulator)
    assert rc == 0, "oracle capacity"
    n = int(rp[-1])
    return rp, col[:n], val[:n], ab[:n]


def _pieces(A, B, rows: np.ndarray, threads: int):
    """The row list split into `threads` contiguous pieces of about equal products."""
    ip = row_ip(A, B, rows)
    cum = np.cumsum(ip)
    cuts = np.searchsorted(cum, np.linspace(0, cum[-1], threads + 1)[1:-1])
    return np.split(rows, cuts)


def row_nnz(A, B, rows=None, threads: int = 1) -> np.ndarray:
    """Distinct columns of each listed row of C = A*B (all rows when rows is None)."""
    lib = _load()
    rows = np.arange(A.rows, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    assert A.cols == B.rows

    def one(r):
        out = np.zeros(len(r), dtype=np.int64)
        lib.oracle_row_nnz(_ptr(A.row_ptr), _ptr(A.col), _ptr(B.row_ptr), _ptr(B.col), B.cols, _ptr(r), len(r),
                           _ptr(out))
        return out
    if threads <= 1 or len(rows) < 2 * threads:
        return one(rows)
    with ThreadPoolExecutor(threads) as ex:
        return np.concatenate(list(ex.map(one, _pieces(A, B, rows, threads))))


def spgemm_rows(A, B, rows, threads: int = 1, accumulator: str = "map"):
    """Rows ``rows`` of C = A*B as (row_ptr local to the list, col, val, abs_sum).  The
    accumulator is the ordered map ("map") or the dense array ("dense"); both give the same
    bits."""
    rows = np.ascontiguousarray(rows, np.int64)
    assert A.cols == B.rows
    if threads <= 1 or len(rows) < 2 * threads:
        return _rows_one(A, B, rows, accumulator)
    pieces = _pieces(A, B, rows, threads)
    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(lambda r: _rows_one(A, B, r, accumulator), pieces))
    rp = [np.zeros(1, np.int64)]
    base = 0
    for p in parts:
        rp.append(p[0][1:] + base)
        base += int(p[0][-1])
    return (np.concatenate(rp), np.concatenate([p[1] for p in parts]),
            np.concatenate([p[2] for p in parts]), np.concatenate([p[3] for p in parts]))


def spgemm(A, B, threads: int = 1, accumulator: str = "map"):
    """Full C = A*B: returns (CSR C, abs_sum per entry)."""
    from synth import CSR  # container only
    rp, col, val, ab = spgemm_rows(A, B, np.arange(A.rows, dtype=np.int64), threads, accumulator)
    return CSR(A.rows, B.cols, rp, col, val), ab
