"""GPU parity of the estimated light-row workflows (Ocean page: HyperLogLog estimation, the
upper-bound method, Table 1 selection, overflow fallback) against the oracles: the HyperLogLog
capacities element by element against oracle/hll.py, and C against the Gustavson oracle under
every workflow, including forced overflow of every estimated row."""
import numpy as np
import pytest

import oracle
import synth
from oracle import hll
from _helpers import compare_full, gpu_product

pytestmark = pytest.mark.gpu


def opts(**kw):
    import sparse_gemm_irregular_gb300 as sg
    return sg.options(**kw)


def dense_overlap(rows, seed):
    """Rows of A with 30 entries over B rows of 80 entries among 100 columns: many products per
    output entry (compression ratio well above 8)."""
    A = synth.random_sparse(rows, 400, 30 / 400, seed)
    B = synth.random_sparse(400, 100, 0.8, seed + 1)
    return A, B


CASES = {
    "random_dup": lambda: (synth.random_sparse(300, 257, 0.03, 1, duplicates=True, empty_rows=True, sort_rows=False),
                           synth.random_sparse(257, 411, 0.05, 51, duplicates=True, empty_rows=True)),
    "rmat12": lambda: (synth.rmat(12, 16, seed=8), None),
    "band": lambda: (synth.banded(20000, 3, seed=2), None),
    "uniform": lambda: (synth.uniform_rows(2048, 8, seed=4), None),
    "overlap": lambda: dense_overlap(500, 6),
}


@pytest.mark.parametrize("case", ["random_dup", "rmat12", "overlap"])
@pytest.mark.parametrize("m", [32, 64])
def test_hll_capacities_match_oracle(gpu_lib, case, m):
    import torch
    import sparse_gemm_irregular_gb300 as sg
    A, B = CASES[case]()
    B = A if B is None else B
    dA = sg.DeviceCSR.from_host(A)
    dB = dA if B is A else sg.DeviceCSR.from_host(B)
    for coef in (hll.coefficient(m), 0.37):
        cap = torch.empty(A.rows, dtype=torch.int64, device="cuda")
        sg.spgemm_hll_estimate(dA.desc(), dB.desc(), m, coef, cap.data_ptr())
        torch.cuda.synchronize()
        expect = hll.capacities(A, B, m, coef, oracle.row_ip(A, B))
        got = cap.cpu().numpy()
        bad = np.nonzero(got != expect)[0]
        assert len(bad) == 0, "row %d: gpu %d oracle %d" % (bad[0], got[bad[0]], expect[bad[0]])


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("wf,kw", [(1, {}), (2, {}), (2, dict(hll_coef=0.05)), (2, dict(hll_registers=32)),
                                   (3, {})])
def test_workflow_parity(gpu_lib, case, wf, kw):
    A, B = CASES[case]()
    B = A if B is None else B
    rp, col, val, st = gpu_product(A, B, opts(workflow=wf, **kw))
    compare_full(A, B, rp, col, val)
    if wf in (1, 2):
        assert st.workflow == wf
    if wf == 2 and kw.get("hll_coef") == 0.05 and st.rows_light > st.rows_dense_light:
        assert st.rows_overflow > 0  # capacities far below the sizes: the fallback pass ran


def test_auto_selection_follows_table_1(gpu_lib):
    # fewer than 64 products per row on average: the upper bound
    A = synth.banded(20000, 3, seed=2)
    assert gpu_product(A, A, opts(workflow=3))[3].workflow == 1
    # 64 products per row but C barely compresses: exact symbolic pass
    A = synth.uniform_rows(2048, 8, seed=4)
    assert gpu_product(A, A, opts(workflow=3))[3].workflow == 0
    # expansion and compression ratios both far above 8: HyperLogLog estimates
    A, B = dense_overlap(800, 9)
    st = gpu_product(A, B, opts(workflow=3))[3]
    assert st.workflow == 2 and st.hll_registers == 64


@pytest.mark.parametrize("wf", [1, 2])
def test_workflow_row_windows_and_host_output(gpu_lib, wf):
    """numeric_rows windows and the host-streamed numeric phase copy the light rows out of their
    temporary slots per window."""
    import torch
    import sparse_gemm_irregular_gb300 as sg
    A = synth.rmat(12, 16, seed=8)
    dA = sg.DeviceCSR.from_host(A)
    p = sg.Product(dA, dA, opts=opts(workflow=wf, tau=512, chunk_width=256, hll_coef=0.5))
    try:
        rp, nnz = p.symbolic()
        full_c, full_v = p.numeric()
        rph = rp.cpu().numpy()
        compare_full(A, A, rph, full_c.cpu().numpy(), full_v.cpu().numpy())
        for b, e in [(0, 1), (37, 2000), (4000, 4096)]:
            n = int(rph[e] - rph[b])
            c = torch.empty(max(n, 1), dtype=torch.int32, device="cuda")
            v = torch.empty(max(n, 1), dtype=torch.float64, device="cuda")
            p.numeric_rows(b, e, c, v)
            torch.cuda.synchronize()
            assert torch.equal(c[:n], full_c[rph[b]:rph[e]])
            assert torch.allclose(v[:n], full_v[rph[b]:rph[e]], rtol=1e-12, atol=0)
        hc = torch.empty(max(nnz, 1), dtype=torch.int32).pin_memory()
        hv = torch.empty(max(nnz, 1), dtype=torch.float64).pin_memory()
        p.numeric_host(hc, hv, window_nnz=5000)
        assert np.array_equal(hc.numpy()[:nnz], full_c.cpu().numpy())
        # repeated numeric into the same arrays: captured, then replayed from a CUDA graph
        for _ in range(3):
            p.numeric(full_c, full_v)
        assert p.stats().numeric_graph == 1
        torch.cuda.synchronize()
        compare_full(A, A, rph, full_c.cpu().numpy(), full_v.cpu().numpy())
    finally:
        p.close()


def test_invalid_workflow_options(gpu_lib):
    import sparse_gemm_irregular_gb300 as sg
    A = synth.random_sparse(20, 20, 0.2, 1)
    dA = sg.DeviceCSR.from_host(A)
    for kw in (dict(workflow=4), dict(workflow=2, hll_registers=48), dict(workflow=2, hll_coef=-1.0)):
        with pytest.raises(sg.SpgemmError) as e:
            sg.Product(dA, dA, opts=opts(**kw))
        assert e.value.code == -1
