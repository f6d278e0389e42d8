"""CPU oracle for C = A * B (TEST INFRASTRUCTURE ONLY).

Used by tests/, the smoke check and the benchmark's CPU-baseline leg; the library never
imports it.  The arithmetic lives in gustavson.cpp: a single-threaded Gustavson product
with an ordered-map accumulator per row (gMAGNUS page, section II-B, Eq. (1),
Algorithm 1).  ``spgemm_rows`` may split a row list across host threads; every thread
runs the same unchanged per-row routine on its own rows.

Parity status: pinned (tests/test_oracle.py) against dense brute force on small inputs,
closed forms (A*I = A, permutations, banded squares, disjoint structure), integer-valued
exact sums and the printed chunk tables do not apply here (they pin the planner).
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


def _rows_one(A, B, rows: np.ndarray):
    lib = _load()
    cap = int(row_ip(A, B, rows).sum())
    rp = np.zeros(len(rows) + 1, dtype=np.int64)
    col = np.zeros(max(cap, 1), dtype=np.int32)
    val = np.zeros(max(cap, 1), dtype=np.float64)
    ab = np.zeros(max(cap, 1), dtype=np.float64)
    rc = lib.oracle_rows(_ptr(A.row_ptr), _ptr(A.col), _ptr(A.val), _ptr(B.row_ptr), _ptr(B.col),
                         _ptr(B.val), _ptr(rows), len(rows), cap, _ptr(rp), _ptr(col), _ptr(val),
                         _ptr(ab))
    assert rc == 0, "oracle capacity"
    n = int(rp[-1])
    return rp, col[:n], val[:n], ab[:n]


def spgemm_rows(A, B, rows, threads: int = 1):
    """Rows ``rows`` of C = A*B as (row_ptr local to the list, col, val, abs_sum)."""
    rows = np.ascontiguousarray(rows, np.int64)
    assert A.cols == B.rows
    if threads <= 1 or len(rows) < 2 * threads:
        return _rows_one(A, B, rows)
    # balance the pieces by intermediate products
    ip = row_ip(A, B, rows)
    cum = np.cumsum(ip)
    cuts = np.searchsorted(cum, np.linspace(0, cum[-1], threads + 1)[1:-1])
    pieces = np.split(rows, cuts)
    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(lambda r: _rows_one(A, B, r), pieces))
    rp = [np.zeros(1, np.int64)]
    base = 0
    for p in parts:
        rp.append(p[0][1:] + base)
        base += int(p[0][-1])
    return (np.concatenate(rp), np.concatenate([p[1] for p in parts]),
            np.concatenate([p[2] for p in parts]), np.concatenate([p[3] for p in parts]))


def spgemm(A, B, threads: int = 1):
    """Full C = A*B: returns (CSR C, abs_sum per entry)."""
    from synth import CSR  # container only
    rp, col, val, ab = spgemm_rows(A, B, np.arange(A.rows, dtype=np.int64), threads)
    return CSR(A.rows, B.cols, rp, col, val), ab
