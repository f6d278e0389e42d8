"""HyperLogLog row-size estimates for C = A * B (TEST INFRASTRUCTURE ONLY).

Used by tests/ and nothing else; the library never imports it.  Plain numpy, written from
the Ocean page ("Ocean: Fast Estimation-Based Sparse General Matrix-Matrix Multiplication on
GPU"): HyperLogLog background (m registers; an element's hash picks its register by the low
bits and offers the rank of the remaining bits, the position of their first set bit; a
register keeps the largest rank offered; the estimate is a bias-corrected harmonic mean of
2^-register) and the construct-and-merge scheme of Figure 3 (one sketch per row of B; the
sketch of row i of C is the element-wise maximum of the sketches of the rows of B that row i
of A selects).  The estimator constants and the small-range (linear counting) correction
follow Flajolet et al. (2007), which the page cites.  Capacities follow the page's overflow
evaluation: estimate x 1.5 (x 2.0 with 32 registers), rounded up.

Readings where the page is silent: the hash is the 32-bit MurmurHash3 finaliser of the
column index (the page names no hash); the register index is its low log2(m) bits and the
rank is counted on the remaining 32 - log2(m) bits (all zero: 33 - log2(m)); a capacity never
exceeds the row's intermediate-product count, which bounds its nnz exactly.

Parity status: pinned (tests/test_oracle_hll.py): rank and index against a bit-string
definition, sketch merging against the sketch of the exact column set of C's rows from the
Gustavson oracle, the estimator against closed forms (empty set, one element), its constant
alpha_m against the integral that defines it, its mean over 2000 seeded sets (unbiased within
1%) and known cardinalities within its stated 1.04/sqrt(m) error, and the capacities (the
ceiling of coefficient x estimate, capped at IP) on rows worked by hand.
"""
from __future__ import annotations

import math

import numpy as np

# alpha_m of the HyperLogLog estimator for the register counts the page uses
ALPHA = {16: 0.673, 32: 0.697, 64: 0.709}


def mix32(c: np.ndarray) -> np.ndarray:
    """MurmurHash3's 32-bit finaliser, applied to each column index (uint32 arithmetic)."""
    h = np.asarray(c, dtype=np.int64).astype(np.uint32)
    h = h ^ (h >> np.uint32(16))
    h = (h.astype(np.uint64) * np.uint64(0x85EBCA6B) & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    h = h ^ (h >> np.uint32(13))
    h = (h.astype(np.uint64) * np.uint64(0xC2B2AE35) & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    h = h ^ (h >> np.uint32(16))
    return h


def index_rank(cols: np.ndarray, m: int):
    """Register index (low bits of the hash) and rank (1 + leading zeros of the other bits)."""
    b = int(m).bit_length() - 1
    assert 1 << b == m
    h = mix32(cols)
    idx = (h & np.uint32(m - 1)).astype(np.int64)
    w = (h >> np.uint32(b)).astype(np.int64)  # 32 - b significant bits
    width = 32 - b
    bl = np.zeros(len(w), dtype=np.int64)  # bit length of w
    for k in range(width):
        bl = np.where((w >> k) != 0, k + 1, bl)
    rank = width - bl + 1
    return idx, rank


def sketch(cols: np.ndarray, m: int) -> np.ndarray:
    """Registers (uint8, m) of one set of column indices."""
    regs = np.zeros(m, dtype=np.int64)
    if len(cols):
        idx, rank = index_rank(np.asarray(cols), m)
        np.maximum.at(regs, idx, rank)
    return regs.astype(np.uint8)


def sketch_rows(B, m: int) -> np.ndarray:
    """One sketch per row of B: uint8 array (B.rows, m)."""
    out = np.zeros((B.rows, m), dtype=np.int64)
    if B.nnz:
        rows = np.repeat(np.arange(B.rows), np.diff(B.row_ptr))
        idx, rank = index_rank(B.col, m)
        np.maximum.at(out, (rows, idx), rank)
    return out.astype(np.uint8)


def merge_rows(A, sk_b: np.ndarray) -> np.ndarray:
    """Sketch of every row of C = A * B: the element-wise maximum over the rows of B selected
    by the row of A (Figure 3 of the Ocean page)."""
    m = sk_b.shape[1]
    out = np.zeros((A.rows, m), dtype=np.uint8)
    for i in range(A.rows):
        a, b = int(A.row_ptr[i]), int(A.row_ptr[i + 1])
        if b > a:
            out[i] = sk_b[A.col[a:b]].max(axis=0)
    return out


def estimate(regs: np.ndarray) -> float:
    """HyperLogLog cardinality estimate of one sketch, with linear counting below 5m/2."""
    regs = np.asarray(regs, dtype=np.int64)
    m = len(regs)
    z = math.fsum(2.0 ** (-int(r)) for r in regs)
    e = ALPHA[m] * m * m / z
    v = int((regs == 0).sum())
    if e <= 2.5 * m and v > 0:
        e = m * math.log(m / v)
    return e


def coefficient(m: int) -> float:
    """Capacity coefficient of the page's overflow evaluation: 2.0 with 32 registers, else 1.5."""
    return 2.0 if m <= 32 else 1.5


def registers_for(ip_total: int, nnz_a: int) -> int:
    """32 registers when the expansion ratio (products per entry of A) is below 48, else 64."""
    er = ip_total / nnz_a if nnz_a else 0.0
    return 32 if er < 48 else 64


def capacities(A, B, m: int, coef: float, ip: np.ndarray) -> np.ndarray:
    """Per-row output capacity: min(IP, ceil(coef * estimate)); 0 for rows without products."""
    sk = merge_rows(A, sketch_rows(B, m))
    cap = np.zeros(A.rows, dtype=np.int64)
    for i in range(A.rows):
        if ip[i] > 0:
            cap[i] = min(int(ip[i]), int(math.ceil(coef * estimate(sk[i]))))
    return cap
