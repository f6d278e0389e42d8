"""Pins for the oracle's Markov-clustering step (Trident page, section 5.7: expansion, column
normalization, pruning below a threshold, element-wise square)."""
import numpy as np
import pytest

import synth
from oracle import mcl
from synth import CSR


def dense(m):
    d = np.zeros((m.rows, m.cols))
    rows = np.repeat(np.arange(m.rows), np.diff(m.row_ptr))
    np.add.at(d, (rows, m.col), m.val)
    return d


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("thr", [0.002, 0.05])
def test_step_matches_dense_computation(seed, thr):
    M = synth.mcl_matrix(7, 4, seed=seed)
    out, amb, C, _ = mcl.step(M, thr)
    D = dense(M)
    E = D @ D
    s = E.sum(axis=0)
    N = np.divide(E, s, out=np.zeros_like(E), where=s > 0)
    present = dense(CSR(C.rows, C.cols, C.row_ptr, C.col, np.ones(C.nnz))) > 0
    # entries on the threshold (values 1/colcount can hit it exactly) may go either way
    on_edge = dense(CSR(C.rows, C.cols, C.row_ptr, C.col, amb.astype(np.float64))) > 0
    keep = present & (N >= thr)
    got = dense(out)
    assert np.array_equal((got > 0) & ~on_edge, keep & ~on_edge)
    both = (got > 0) & keep
    assert np.allclose(got[both], N[both] ** 2, rtol=1e-13, atol=0)


def test_permutation_is_a_fixed_point():
    n = 50
    perm = np.random.default_rng(3).permutation(n)
    P = CSR(n, n, np.arange(n + 1, dtype=np.int64), perm.astype(np.int32), np.ones(n))
    out, _, _, _ = mcl.step(P, 0.002)
    # P*P is a permutation; its columns already sum to 1; nothing pruned; 1^2 = 1
    assert np.array_equal(out.col, perm[perm].astype(np.int32)) and np.all(out.val == 1.0)


@pytest.mark.parametrize("k", [2, 5, 8])
def test_block_uniform_stochastic_closed_form(k):
    # blockdiag of (1/k) J_k: idempotent under squaring, columns sum to 1, every entry 1/k
    blocks = 4
    n = k * blocks
    r, c = np.divmod(np.arange(n * k), k)
    cols = (r // k) * k + c
    M = CSR(n, n, np.arange(0, n * k + 1, k, dtype=np.int64), cols.astype(np.int32), np.full(n * k, 1.0 / k))
    out, _, _, _ = mcl.step(M, 0.002)
    assert out.nnz == n * k and np.allclose(out.val, 1.0 / k ** 2, rtol=1e-15)
    pruned, _, _, _ = mcl.step(M, 1.0 / k + 1e-9)  # every normalized entry (1/k) lies below
    assert pruned.nnz == 0
