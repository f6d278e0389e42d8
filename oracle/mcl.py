"""One Markov-clustering iteration (TEST INFRASTRUCTURE ONLY; the library never imports it).

Plain numpy around the Gustavson oracle, in the order the Trident page gives for MCL (section
5.7): the expansion C = M * M, then normalize every column of C to sum 1, prune the entries
below the threshold, and square the remaining entries element-wise.  Column sums are correctly
rounded (math.fsum).  An entry is kept when C[i,j] / colsum_j >= threshold.

`ambiguous` marks the entries whose normalized value lies within a relative `band` of the
threshold: there the keep decision depends on the last bits of the column sum, which differ with
the summation order, so either decision is correct.

Parity status: pinned (tests/test_oracle_mcl.py) against a dense numpy computation of the same
step on small matrices, against permutation matrices (a fixed point of the step) and against
block-uniform stochastic matrices (idempotent under the expansion, closed-form values).
"""
from __future__ import annotations

import math

import numpy as np

from . import spgemm


def step(M, threshold: float, threads: int = 1, band: float = 1e-10):
    """Returns (new CSR, ambiguous mask over C's entries, C, normalized values of C)."""
    from synth import CSR  # container only
    C, _ = spgemm(M, M, threads=threads)
    sums = np.zeros(C.cols)
    order = np.argsort(C.col, kind="stable")
    cols_sorted = C.col[order]
    vals_sorted = C.val[order]
    bounds = np.searchsorted(cols_sorted, np.arange(C.cols + 1))
    for j in range(C.cols):
        a, b = bounds[j], bounds[j + 1]
        if b > a:
            sums[j] = math.fsum(vals_sorted[a:b])
    norm = np.zeros(C.nnz)
    if C.nnz:
        norm = C.val / sums[C.col]
    keep = norm >= threshold
    ambiguous = np.abs(norm - threshold) <= band * threshold
    rows = np.repeat(np.arange(C.rows), np.diff(C.row_ptr))
    counts = np.bincount(rows[keep], minlength=C.rows).astype(np.int64)
    rp = np.zeros(C.rows + 1, dtype=np.int64)
    np.cumsum(counts, out=rp[1:])
    out = CSR(C.rows, C.cols, rp, C.col[keep].astype(np.int32), norm[keep] ** 2)
    return out, ambiguous, C, norm
