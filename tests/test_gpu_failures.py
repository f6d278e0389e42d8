"""Failure detection on the GPU without faulting it: every failure is made on purpose through an
option, reported as a status code by the call that synchronises, and the device stays usable --
the next product on it matches the oracle.

  * a workspace budget too small for the product  -> SPGEMM_ERR_OUT_OF_MEMORY, clean destroy;
  * light-row hash tables capped below the rows' sizes -> the bounded probe gives up,
    SPGEMM_ERR_DEVICE;
  * the staged multisplit's first bulk-copy wait allowed a single poll -> the wait runs out, the
    block records the timeout, waits (bounded) for its own copies in flight and returns,
    SPGEMM_ERR_DEVICE."""
import numpy as np
import pytest

import synth
from _helpers import compare_full, gpu_product

pytestmark = pytest.mark.gpu


def _flags(msg):
    """The device error word named in a failure message ("... device check failed (flags 0x..)")."""
    import re
    m = re.search(r"flags 0x([0-9a-f]+)", msg)
    assert m, msg
    return int(m.group(1), 16)


def _next_product_ok():
    A = synth.rmat(12, 16, seed=21)
    rp, col, val, _ = gpu_product(A, A)
    compare_full(A, A, rp, col, val)


def test_workspace_budget_out_of_memory(gpu_lib):
    import torch
    import sparse_gemm_irregular_gb300 as sg
    A = synth.rmat(12, 16, seed=8)
    dA = sg.DeviceCSR.from_host(A)
    def run(limit):
        p = None
        try:
            p = sg.Product(dA, dA, opts=sg.options(workspace_limit=limit, tau=512, chunk_width=256))
            p.symbolic()
            p.numeric()
        finally:
            if p is not None:
                p.close()
    for limit in (64 * 1024, 4 << 20):   # fails in create, and later (symbolic or numeric)
        with pytest.raises(sg.SpgemmError) as e:
            run(limit)
        assert e.value.code == sg.binding.ERRORS_BY_NAME["OUT_OF_MEMORY"], sg.spgemm_last_error()
    torch.cuda.synchronize()
    # a budget that fits runs to the end and matches the oracle
    p = sg.Product(dA, dA, opts=sg.options(workspace_limit=1 << 33, tau=512, chunk_width=256))
    try:
        rp, nnz = p.symbolic()
        col, val = p.numeric()
        torch.cuda.synchronize()
        compare_full(A, A, rp.cpu().numpy(), col.cpu().numpy()[:nnz], val.cpu().numpy()[:nnz])
    finally:
        p.close()
    _next_product_ok()


def test_hash_table_overflow_reported(gpu_lib):
    import sparse_gemm_irregular_gb300 as sg
    A = synth.random_sparse(500, 400, 0.05, 3)                  # about 20 entries per row
    B = synth.random_sparse(400, 3000, 0.02, 4)                 # about 60 per row: rows of ~1000 columns
    dA, dB = sg.DeviceCSR.from_host(A), sg.DeviceCSR.from_host(B)
    flags = sg.binding.FLAG_NO_ESC | sg.binding.FLAG_NO_DENSE_LIGHT
    p = sg.Product(dA, dB, opts=sg.options(flags=flags, debug_hash_slots=64))
    try:
        with pytest.raises(sg.SpgemmError) as e:
            p.symbolic()
        assert e.value.code == sg.binding.ERRORS_BY_NAME["DEVICE"]
        assert _flags(sg.spgemm_last_error()) & 0x1  # the hash-table-full bit
    finally:
        p.close()
    _next_product_ok()


def test_staged_multisplit_wait_timeout(gpu_lib):
    """The first bulk-copy wait of every block of the staged multisplit gets one poll: it runs
    out while its copy is in flight, the block drains and returns, and the call reports a
    device-side failure instead of hanging or faulting."""
    import sparse_gemm_irregular_gb300 as sg
    A = synth.rmat(13, 16, seed=6)
    dA = sg.DeviceCSR.from_host(A)
    kw = dict(flags=sg.binding.FLAG_TMA_SPLIT, tau=256, chunk_width=64, chunks_max=4)
    p = sg.Product(dA, dA, opts=sg.options(debug_wait_spins=1, **kw))
    try:
        with pytest.raises(sg.SpgemmError) as e:
            p.symbolic()
        assert e.value.code == sg.binding.ERRORS_BY_NAME["DEVICE"]
        assert _flags(sg.spgemm_last_error()) & 0x10  # the timeout bit
    finally:
        p.close()
    # the same product with the normal limit is correct
    rp, col, val, st = gpu_product(A, A, sg.options(**kw))
    assert st.levels_run >= 2
    compare_full(A, A, rp, col, val, threads=8)
    _next_product_ok()
