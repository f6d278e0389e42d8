"""GPU parity of the Markov-clustering iteration (Trident page, section 5.7: expansion on the
library's SpGEMM, column normalization, pruning below 0.002, element-wise square) against the
oracle, one iteration at a time from the oracle's previous matrix.  Keep decisions are compared
exactly except on entries whose normalized value lies within 1e-10 (relative) of the threshold,
where the column sum's summation order decides and either outcome is correct; kept values agree
within 1e-11 relative (C within 1e-12, column sums of positive terms within n*eps, squared)."""
import numpy as np
import pytest

import synth
from oracle import mcl

pytestmark = pytest.mark.gpu


def keys(rows_ptr, col, ncols):
    r = np.repeat(np.arange(len(rows_ptr) - 1, dtype=np.int64), np.diff(rows_ptr))
    return r * ncols + col.astype(np.int64)


@pytest.mark.parametrize("scale,ef,thr", [(10, 8, 0.002), (11, 16, 0.002), (9, 4, 0.05)])
def test_mcl_iterations(gpu_lib, scale, ef, thr):
    import sparse_gemm_irregular_gb300 as sg
    M = synth.mcl_matrix(scale, ef, seed=scale)
    for it in range(3):
        ref, amb, C, norm = mcl.step(M, thr, threads=8)
        out = sg.mcl_iteration(sg.DeviceCSR.from_host(M), thr)
        rp, col, val = out.to_host()
        n = M.cols
        kg = keys(rp, col, n)
        kc = keys(C.row_ptr, C.col, n)
        kamb = set(kc[amb].tolist())
        kref = keys(ref.row_ptr, ref.col, n)
        sg_set, ref_set = set(kg.tolist()), set(kref.tolist())
        assert sg_set <= set(kc.tolist())
        assert sg_set - kamb == ref_set - kamb, "iteration %d: keep decisions differ" % it
        # rows sorted like C, values of the entries both kept
        common = np.isin(kg, kref)
        pos = np.searchsorted(kref, kg[common])
        assert np.allclose(val[common], ref.val[pos], rtol=1e-11, atol=0)
        M = ref
        if M.nnz == 0:
            break


def test_mcl_prune_edge_cases(gpu_lib):
    import torch
    import sparse_gemm_irregular_gb300 as sg
    from synth import CSR
    # empty matrix and a zero threshold (keeps everything: normalized values are positive)
    Z = CSR(5, 5, np.zeros(6, np.int64), np.zeros(0, np.int32), np.zeros(0))
    out = sg.mcl_iteration(sg.DeviceCSR.from_host(Z), 0.002)
    assert out.nnz == 0 and torch.all(out.row_ptr == 0)
    M = synth.mcl_matrix(8, 4, seed=2)
    ref, _, C, norm = mcl.step(M, 0.0)
    out = sg.mcl_iteration(sg.DeviceCSR.from_host(M), 0.0)
    assert out.nnz == C.nnz
    with pytest.raises(sg.SpgemmError):
        sg.spgemm_mcl_prune_symbolic(sg.DeviceCSR.from_host(M).desc(), -1.0, 0, 0)
