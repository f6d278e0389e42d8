"""spgemm_symbolic_noalloc: the row sizes of C for callers that cannot allocate device memory
(code inside an allocator or memory manager, loops that forbid allocation after start-up).
It must give the same C.row_ptr and nnz as spgemm_symbolic, call after call, although every
call reuses one static device array.  This file sorts last so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def _symbolic_reference(A, B):
    import sparse_gemm_irregular_gb300 as sg
    dA = sg.DeviceCSR.from_host(A)
    dB = sg.DeviceCSR.from_host(B)
    p = sg.Product(dA, dB)
    rp, nnz = p.symbolic()
    out = rp.cpu().numpy(), nnz
    p.close()
    return dA, dB, out


@pytest.mark.parametrize("case", ["uniform", "band", "random_rect"])
def test_noalloc_matches_symbolic_twice(case):
    import torch
    import sparse_gemm_irregular_gb300 as sg
    from sparse_gemm_irregular_gb300 import binding
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    if case == "uniform":
        A = B = synth.config(1)
    elif case == "band":
        A = B = synth.banded(200_000, 3)
    else:
        A = synth.random_sparse(5000, 3000, 0.002, 11, duplicates=True, empty_rows=True, sort_rows=False)
        B = synth.random_sparse(3000, 7000, 0.003, 12, duplicates=True, sort_rows=False)
    dA, dB, (ref_rp, ref_nnz) = _symbolic_reference(A, B)
    da, db = dA.desc(), dB.desc()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):  # the static array keeps the previous call's contents
        rp = torch.full((A.rows + 1,), -7, dtype=torch.int64, device="cuda")
        nnz = binding.spgemm_symbolic_noalloc(A.rows, A.cols, B.cols, da, db, rp.data_ptr(), stream)
        assert nnz == ref_nnz
        assert np.array_equal(rp.cpu().numpy(), ref_rp)


def test_noalloc_rejects_limits():
    import torch
    import sparse_gemm_irregular_gb300 as sg
    from sparse_gemm_irregular_gb300 import binding
    lib = sg.load()
    # more rows than the static array covers: rejected before any GPU work
    big = binding.spgemm_csr(1 << 25, 4, 0, 1, 0, 0)
    b4 = binding.spgemm_csr(4, 4, 0, 1, 0, 0)
    nnz = ctypes.c_int64()
    rc = lib.spgemm_symbolic_noalloc(1 << 25, 4, 4, ctypes.byref(big), ctypes.byref(b4), ctypes.c_void_p(1),
                                     ctypes.byref(nnz), None)
    assert rc == -1 and "16,777,215" in sg.spgemm_last_error()
    # a row with more than 2048 intermediate products is reported after the kernels ran
    A = synth.random_sparse(8, 64, 1.0, 3)            # 64 entries per row
    B = synth.random_sparse(64, 4096, 0.02, 4)        # ~80 per row -> ~5000 IP per row
    dA, dB = sg.DeviceCSR.from_host(A), sg.DeviceCSR.from_host(B)
    rp = torch.empty(A.rows + 1, dtype=torch.int64, device="cuda")
    with pytest.raises(sg.SpgemmError) as e:
        binding.spgemm_symbolic_noalloc(A.rows, A.cols, B.cols, dA.desc(), dB.desc(), rp.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)
    assert e.value.code == -1
    # and the next valid call is not affected by the flag left behind
    C = synth.config(1)
    dC, _, (ref_rp, ref_nnz) = _symbolic_reference(C, C)
    rp = torch.empty(C.rows + 1, dtype=torch.int64, device="cuda")
    nnz = binding.spgemm_symbolic_noalloc(C.rows, C.cols, C.cols, dC.desc(), dC.desc(), rp.data_ptr(),
                                          torch.cuda.current_stream().cuda_stream)
    assert nnz == ref_nnz and np.array_equal(rp.cpu().numpy(), ref_rp)
