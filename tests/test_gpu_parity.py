"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element by element.

Small and medium inputs are compared in full; the full-size workloads of the benchmark are
compared on a sample of rows (all the heaviest rows plus a seeded uniform sample) and through
invariants that hold at any size.  Planner overrides force the rare paths on small inputs:
every row heavy, several multisplit levels, light chunks at early levels, recomputation across
many heavy batches."""
import numpy as np
import pytest

import oracle
import synth
from _helpers import (compare_full, compare_rows, compare_sampled_device, device_invariants,
                      gpu_product, gpu_product_device, invariants, release_device_memory)

pytestmark = pytest.mark.gpu


def opts(**kw):
    import sparse_gemm_irregular_gb300 as sg
    return sg.options(**kw)


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("dup,empty,sort", [(False, False, True), (True, True, False)])
def test_small_random_default(gpu_lib, seed, dup, empty, sort):
    A = synth.random_sparse(300, 257, 0.03, seed, duplicates=dup, empty_rows=empty, sort_rows=sort)
    B = synth.random_sparse(257, 411, 0.05, seed + 50, duplicates=dup, empty_rows=empty, sort_rows=sort)
    rp, col, val, st = gpu_product(A, B)
    compare_full(A, B, rp, col, val)


FORCED = [
    # every row heavy, one level of 8 chunks of width 64
    dict(flags=1, tau=64, chunk_width=64, chunks_max=8),
    # heavy above 16, two levels (4 x 4 chunks of width 32), light chunks at level 0
    dict(tau=16, chunk_width=32, chunks_max=4),
    # four levels of 2 chunks
    dict(tau=8, chunk_width=32, chunks_max=2),
    # everything heavy, one chunk per row (W covers all columns)
    dict(flags=1, tau=32, chunk_width=512),
    # many heavy batches, recomputed in the numeric phase
    dict(tau=16, chunk_width=64, chunks_max=4, heavy_batch_elems=700, flags=16),
    # light rows only, hash accumulators
    dict(flags=2 | 4, tau=4096),
    # direct split of level 0 (outer product writes C^_reord), one level of 8 chunks
    dict(flags=256, tau=16, chunk_width=64, chunks_max=16),
    dict(flags=256 | 1, tau=64, chunk_width=64, chunks_max=8),
    dict(flags=256 | 16, tau=16, chunk_width=64, chunks_max=16, heavy_batch_elems=700),
    # bulk-copy staged multisplit: two levels, and four levels with recompute batches
    dict(flags=512, tau=16, chunk_width=32, chunks_max=4),
    dict(flags=512 | 16, tau=8, chunk_width=32, chunks_max=2, heavy_batch_elems=700),
    # level-0 histogram counted per product inside the outer product
    dict(flags=1024, tau=16, chunk_width=32, chunks_max=4),
    dict(flags=1024 | 16, tau=8, chunk_width=32, chunks_max=2, heavy_batch_elems=700),
    # short hash rows in the shared hash tables instead of expand-sort-compact
    dict(flags=4096),
    dict(flags=4096 | 2 | 4, tau=4096),
    # heavy rows generating their products from the column-split B (no C^): one level of 8 chunks,
    # every row heavy, 16 chunks per row, many batches, one chunk per row, hash chunks in warps only
    dict(flags=8192, tau=16, chunk_width=32, chunks_max=4),
    dict(flags=8192 | 1, tau=64, chunk_width=64, chunks_max=8),
    dict(flags=8192, tau=16, chunk_width=32, chunks_max=16),
    dict(flags=8192, tau=16, chunk_width=64, chunks_max=4, heavy_batch_elems=700),
    dict(flags=8192 | 1, tau=32, chunk_width=512),
    dict(flags=8192 | 1, tau=8, chunk_width=16),
]


@pytest.mark.parametrize("kw", FORCED)
@pytest.mark.parametrize("seed", [3, 4])
def test_forced_paths(gpu_lib, kw, seed):
    A = synth.random_sparse(200, 180, 0.06, seed, duplicates=True, empty_rows=True, sort_rows=False)
    B = synth.random_sparse(180, 500, 0.08, seed + 9, duplicates=True, empty_rows=True, sort_rows=False)
    rp, col, val, st = gpu_product(A, B, opts(**kw))
    compare_full(A, B, rp, col, val)
    if kw.get("flags", 0) & 1:
        assert st.rows_heavy == int((oracle.row_ip(A, B) > 0).sum())
    if kw.get("chunks_max") == 2:
        assert st.levels_run >= 2
    assert st.fused == (1 if kw.get("flags", 0) & 8192 and st.rows_heavy > 0 else 0)


@pytest.mark.parametrize("kw", [dict(), dict(tau=16, chunk_width=32, chunks_max=4),
                                dict(flags=1, tau=64, chunk_width=64, chunks_max=8)])
def test_integer_values_exact(gpu_lib, kw):
    A = synth.random_sparse(150, 160, 0.1, 21, duplicates=True, integer_values=True, sort_rows=False)
    B = synth.random_sparse(160, 300, 0.1, 22, duplicates=True, integer_values=True, sort_rows=False)
    rp, col, val, _ = gpu_product(A, B, opts(**kw) if kw else None)
    orp, ocol, oval, _ = oracle.spgemm_rows(A, B, np.arange(A.rows))
    assert np.array_equal(rp, orp) and np.array_equal(col, ocol)
    assert np.array_equal(val, oval)  # exact integers: any summation order gives the same bits


@pytest.mark.parametrize("flags", [0, 64, 128, 256, 512, 1024, 4096, 8192])
def test_rmat_small_full(gpu_lib, flags):
    """R-MAT scale 14, edge factor 16: heavy rows above the default tau, several chunks per
    row (dense chunks among them), thousands of light rows in every ladder bin -- compared in
    full (multisplit path, plain shared atomics in the multisplit, dense chunks in L2, direct
    split, bulk-copy staged multisplit, per-product level-0 histogram, short hash rows in
    shared hash tables instead of expand-sort-compact, heavy chunks generated from the
    column-split B)."""
    A = synth.rmat(14, 16, seed=5)
    rp, col, val, st = gpu_product(A, A, opts(flags=flags) if flags else None)
    assert st.rows_heavy > 0 and st.rows_light > 0 and st.dense_elems > 0
    compare_full(A, A, rp, col, val, threads=16)


def test_rmat_small_forced_levels(gpu_lib):
    A = synth.rmat(13, 16, seed=6)
    rp, col, val, st = gpu_product(A, A, opts(tau=256, chunk_width=64, chunks_max=4))
    assert st.levels_run >= 2
    compare_full(A, A, rp, col, val, threads=16)


def test_config1_full(gpu_lib):
    A = synth.config(1)
    rp, col, val, _ = gpu_product(A, A)
    compare_full(A, A, rp, col, val)


def test_config2_full(gpu_lib):
    A = synth.config(2)
    rp, col, val, st = gpu_product(A, A)
    assert st.rows_dense_light == A.rows  # the shortened dense path
    assert rp[-1] == 13 * A.rows - 42
    compare_full(A, A, rp, col, val, threads=16)


def test_banded_ones_closed_form(gpu_lib):
    A = synth.banded(100_000, 3)
    A.val = np.ones(A.nnz)
    rp, col, val, _ = gpu_product(A, A)
    assert rp[-1] == 13 * A.rows - 42
    for i in (10, 5000, 99_000):
        a, b = rp[i], rp[i + 1]
        assert np.array_equal(col[a:b], np.arange(i - 6, i + 7))
        assert np.array_equal(val[a:b], 7.0 - np.abs(np.arange(-6, 7)))


def sample_rows(A, B, n_top=300, n_uniform=3000, seed=0):
    ip = oracle.row_ip(A, B)
    top = np.argsort(ip)[-n_top:]
    uni = (synth.draws(seed, synth.STREAM_SAMPLE, 0, n_uniform) % np.uint64(A.rows)).astype(np.int64)
    return np.unique(np.concatenate([top, uni]))


@pytest.mark.parametrize("flags", [0, 256, 8192])
def test_config3_full_size_sampled(gpu_lib, flags):
    A = synth.config(3)
    p, rp, col, val = gpu_product_device(A, A, opts(flags=flags) if flags else None)
    st = p.stats()
    assert st.rows_heavy > 0 and st.resident == (0 if flags & 8192 else 1)
    rowsum, _ = device_invariants(A, A, rp, col, val)
    compare_sampled_device(A, A, rp, col, val, sample_rows(A, A))
    p.close()
    del rp, col, val
    release_device_memory()


@pytest.mark.parametrize("flags", [0, 256, 8192])
def test_config5_full_size_sampled(gpu_lib, flags):
    M = synth.config(5)
    p, rp, col, val = gpu_product_device(M, M, opts(flags=flags) if flags else None)
    st = p.stats()
    assert st.rows_heavy > 0
    _, colsum = device_invariants(M, M, rp, col, val)
    # C = M M is column-stochastic
    assert float((colsum - 1.0).abs().max()) <= 1e-9
    compare_sampled_device(M, M, rp, col, val, sample_rows(M, M, n_top=100, n_uniform=2000))
    p.close()
    del rp, col, val
    release_device_memory()


def test_identity_and_empty(gpu_lib):
    from synth import CSR
    A = synth.random_sparse(64, 64, 0.1, 7)
    I = CSR(64, 64, np.arange(65, dtype=np.int64), np.arange(64, dtype=np.int32), np.ones(64))
    rp, col, val, _ = gpu_product(A, I)
    assert np.array_equal(rp, A.row_ptr) and np.array_equal(col, A.col) and np.array_equal(val, A.val)
    Z = CSR(10, 64, np.zeros(11, np.int64), np.zeros(0, np.int32), np.zeros(0))
    rp, col, val, _ = gpu_product(Z, A)
    assert np.all(rp == 0) and len(col) == 0


def test_numeric_rows_window(gpu_lib):
    import torch
    import sparse_gemm_irregular_gb300 as sg
    A = synth.rmat(12, 16, seed=8)
    dA = sg.DeviceCSR.from_host(A)
    p = sg.Product(dA, dA, opts=opts(tau=512, chunk_width=256))
    rp, nnz = p.symbolic()
    full_c, full_v = p.numeric()
    rph = rp.cpu().numpy()
    for b, e in [(0, 1), (0, 100), (37, 2000), (4000, 4096), (0, 4096)]:
        n = int(rph[e] - rph[b])
        c = torch.empty(max(n, 1), dtype=torch.int32, device="cuda")
        v = torch.empty(max(n, 1), dtype=torch.float64, device="cuda")
        p.numeric_rows(b, e, c, v)
        torch.cuda.synchronize()
        assert torch.equal(c[:n], full_c[rph[b]:rph[e]])
        assert torch.equal(v[:n], full_v[rph[b]:rph[e]]) or torch.allclose(v[:n], full_v[rph[b]:rph[e]], rtol=1e-12)
    p.close()


def test_validate_flag_rejects_bad_column(gpu_lib):
    import sparse_gemm_irregular_gb300 as sg
    A = synth.random_sparse(20, 20, 0.2, 1)
    A.col = A.col.copy()
    A.col[3] = 25  # out of range for 20 columns
    dA = sg.DeviceCSR.from_host(A)
    B = sg.DeviceCSR.from_host(synth.random_sparse(20, 20, 0.2, 2))
    with pytest.raises(sg.SpgemmError) as e:
        sg.Product(dA, B, opts=opts(flags=8))
    assert e.value.code == -2


@pytest.mark.parametrize("case,window", [("rmat", 0), ("rmat", 20000), ("recompute", 3000), ("light", 2000),
                                         ("rmat", 1), ("fused", 3000), ("fused_batches", 3000)])
def test_numeric_host_windows(gpu_lib, case, window):
    """spgemm_numeric_host: C computed in row windows and streamed into pinned host arrays equals
    the oracle -- one window, many windows (down to one row each), recomputed heavy batches
    (windows of whole batches) and light rows only."""
    import torch
    import sparse_gemm_irregular_gb300 as sg
    if case == "rmat":
        A, B, kw = synth.rmat(13, 16, seed=8), None, None
    elif case == "fused":
        A, B, kw = synth.rmat(13, 16, seed=8), None, dict(flags=8192, tau=512, chunk_width=256)
    elif case == "fused_batches":
        A, B, kw = synth.rmat(13, 16, seed=8), None, dict(flags=8192, tau=512, chunk_width=256,
                                                          heavy_batch_elems=200000)
    elif case == "recompute":
        A = synth.random_sparse(200, 180, 0.06, 3, duplicates=True, empty_rows=True, sort_rows=False)
        B = synth.random_sparse(180, 500, 0.08, 12, duplicates=True, empty_rows=True, sort_rows=False)
        kw = dict(tau=16, chunk_width=64, chunks_max=4, heavy_batch_elems=700, flags=16)
    else:
        A = synth.random_sparse(300, 250, 0.05, 5, duplicates=True, empty_rows=True, sort_rows=False)
        B = synth.random_sparse(250, 400, 0.05, 6)
        kw = dict(flags=2 | 4, tau=4096)
    B = A if B is None else B
    dA = sg.DeviceCSR.from_host(A)
    dB = dA if B is A else sg.DeviceCSR.from_host(B)
    p = sg.Product(dA, dB, opts=opts(**kw) if kw else None)
    try:
        _, nnz = p.symbolic()
        rp = torch.empty(A.rows + 1, dtype=torch.int64).pin_memory()
        col = torch.empty(max(nnz, 1), dtype=torch.int32).pin_memory()
        val = torch.empty(max(nnz, 1), dtype=torch.float64).pin_memory()
        p.numeric_host(col, val, rp, window_nnz=window)
        if case == "recompute":
            assert p.stats().resident == 0
    finally:
        p.close()
    compare_full(A, B, rp.numpy(), col.numpy()[:nnz], val.numpy()[:nnz], threads=16)


def test_config4_row_windows(gpu_lib):
    """R-MAT scale 21, edge factor 32: C (about 6e10 entries) fits neither the device nor the
    test host.  The symbolic phase runs at full size (heavy batches recomputed, not resident);
    the numeric phase runs in row windows (spgemm_numeric_rows) -- the heaviest rows, a middle
    block and the last block.  Every window row is checked against C x = A (B x); every window
    row with at most 2e6 intermediate products against the oracle."""
    import torch
    import sparse_gemm_irregular_gb300 as sg
    A = synth.config(4)
    ip = oracle.row_ip(A, A)
    dA = sg.DeviceCSR.from_host(A)
    p = sg.Product(dA, dA)
    try:
        rp, nnz = p.symbolic()
        st = p.stats()
        assert st.rows_heavy > 0 and st.resident == 0
        rp_h = rp.cpu().numpy()
        del rp
        row_nnz = np.diff(rp_h)
        assert rp_h[0] == 0 and rp_h[-1] == nnz and np.all(row_nnz >= 0) and np.all(row_nnz <= ip)
        x = synth.uniform(11, synth.STREAM_SAMPLE, 0, A.cols, 0.0, 1.0)
        brow = np.repeat(np.arange(A.rows), np.diff(A.row_ptr))
        bx = np.bincount(brow, weights=A.val * x[A.col], minlength=A.rows)  # B x (B = A)
        m = A.rows
        checked = 0
        for rb, re in [(0, 32), (m // 2, m // 2 + 8192), (m - 8192, m)]:
            cnt = int(rp_h[re] - rp_h[rb])
            col = torch.empty(max(cnt, 1), dtype=torch.int32, device="cuda")
            val = torch.empty(max(cnt, 1), dtype=torch.float64, device="cuda")
            p.numeric_rows(rb, re, col, val)
            torch.cuda.synchronize()
            c = col.cpu().numpy()[:cnt]
            v = val.cpu().numpy()[:cnt]
            del col, val
            lrp = rp_h[rb:re + 1] - rp_h[rb]
            rid = np.repeat(np.arange(re - rb), np.diff(lrp))
            # sorted, unique columns in every row
            same_row = rid[1:] == rid[:-1]
            assert np.all(c[1:][same_row] > c[:-1][same_row])
            # C x = A (B x), all values nonnegative
            y = np.bincount(rid, weights=v * x[c], minlength=re - rb)
            a0, a1 = A.row_ptr[rb], A.row_ptr[re]
            arid = np.repeat(np.arange(re - rb), np.diff(A.row_ptr[rb:re + 1]))
            ref = np.bincount(arid, weights=A.val[a0:a1] * bx[A.col[a0:a1]], minlength=re - rb)
            assert np.all(np.abs(y - ref) <= 1e-11 * ref + 1e-300)
            rows = np.arange(rb, re)
            small = rows[ip[rows] <= 2_000_000]
            compare_rows(A, A, rp_h - rp_h[rb], c, v, small, threads=16)
            checked += len(small)
        assert checked > 10000
    finally:
        p.close()
        release_device_memory()


@pytest.mark.parametrize("case", ["light", "resident", "recompute", "no_graph", "fused"])
def test_numeric_repeat_graph(gpu_lib, case):
    """Repeated numeric calls into the same arrays: the second call is captured into a CUDA graph
    and later calls replay it, where the phase has no host synchronisation (no heavy row, or
    C^_reord resident).  Without a resident C^_reord each call reads the current values of A and
    B, so new values (same structure) give the oracle's product of the new values."""
    import torch
    import sparse_gemm_irregular_gb300 as sg
    if case == "light":
        A, kw = synth.uniform_rows(2048, 8, seed=3), None
    elif case == "resident":
        A, kw = synth.rmat(12, 16, seed=8), dict(tau=512, chunk_width=256)
    elif case == "recompute":
        A, kw = synth.rmat(11, 16, seed=9), dict(tau=256, chunk_width=128, heavy_batch_elems=20000, flags=16)
    elif case == "fused":
        A, kw = synth.rmat(12, 16, seed=8), dict(tau=512, chunk_width=256, flags=sg.binding.FLAG_FUSED)
    else:
        A, kw = synth.uniform_rows(2048, 8, seed=4), dict(flags=sg.binding.FLAG_NO_GRAPH)
    dA = sg.DeviceCSR.from_host(A)
    p = sg.Product(dA, dA, opts=opts(**kw) if kw else None)
    try:
        rp, nnz = p.symbolic()
        st0 = p.stats()
        if case == "resident":
            assert st0.resident == 1 and st0.rows_heavy > 0
        if case == "recompute":
            assert st0.resident == 0 and st0.heavy_batches > 1
        if case == "fused":
            assert st0.fused == 1 and st0.rows_heavy > 0 and st0.resident == 0
        col = torch.empty(max(nnz, 1), dtype=torch.int32, device="cuda")
        val = torch.empty(max(nnz, 1), dtype=torch.float64, device="cuda")
        graphed, launches = [], []
        for call in range(4):
            if call >= 2 and case != "resident":  # new values, same structure
                vals = synth.uniform(40 + call, 0, 0, A.nnz, -1.0, 1.0)
                A = synth.with_values(A, vals)
                dA.val.copy_(torch.from_numpy(vals))
            k0 = sg.spgemm_kernel_launches()
            p.numeric(col, val)
            torch.cuda.synchronize()
            launches.append(sg.spgemm_kernel_launches() - k0)
            graphed.append(p.stats().numeric_graph)
            compare_full(A, A, rp.cpu().numpy(), col.cpu().numpy()[:nnz], val.cpu().numpy()[:nnz])
        expect = [0, 1, 1, 1] if case in ("light", "resident", "fused") else [0, 0, 0, 0]
        assert graphed == expect, sg.spgemm_last_error()
        # the first call also bins the light rows by their exact size (once per handle); a replay
        # counts the kernels its graph holds
        assert launches[1] == launches[2] == launches[3] > 0 and launches[0] >= launches[1]
        # other output arrays: a new key, so the next call runs eagerly again
        col2, val2 = torch.empty_like(col), torch.empty_like(val)
        p.numeric(col2, val2)
        assert p.stats().numeric_graph == 0
        torch.cuda.synchronize()
        compare_full(A, A, rp.cpu().numpy(), col2.cpu().numpy()[:nnz], val2.cpu().numpy()[:nnz])
    finally:
        p.close()


@pytest.mark.parametrize("case", ["rmat_pair", "a_times_r", "a_times_r_heavy", "a_times_at", "rmat_pair_fused",
                                  "a_times_at_fused"])
def test_general_products(gpu_lib, case):
    """Products beyond C = A*A: an R-MAT pair A*B with B != A, a rectangular A*R with a tall
    aggregation operator R, and A*A^T of a rectangular A (heavy path forced on small inputs)."""
    kw = None
    if case.startswith("rmat_pair"):
        A, B = synth.rmat(13, 16, seed=1), synth.rmat(13, 16, seed=2)
        if case.endswith("fused"):
            kw = dict(tau=256, chunk_width=512, flags=8192)
    elif case.startswith("a_times_r"):
        A = synth.rmat(13, 16, seed=3)
        B = synth.aggregation(A.cols, 700, seed=4, per_row=2)
        if case.endswith("heavy"):
            kw = dict(tau=64, chunk_width=64, chunks_max=4)
    else:
        A = synth.random_sparse(3000, 5000, 0.004, 6, duplicates=True, empty_rows=True, sort_rows=False)
        B = synth.transpose(A)
        kw = dict(tau=128, chunk_width=256, flags=8192 if case.endswith("fused") else 0)
    rp, col, val, st = gpu_product(A, B, opts(**kw) if kw else None)
    compare_full(A, B, rp, col, val, threads=16)
    if kw:
        assert st.rows_heavy > 0


@pytest.mark.parametrize("case", ["config1", "band", "random_dup", "long_a_rows"])
def test_esc_short_rows(gpu_lib, case):
    """Expand-sort-compact (the default for hash rows of at most 64 products) against the hash
    tables: config 1 (64 per row), a band (49, shortened dense either way),
    duplicates and empty rows, and rows of A longer than a warp whose B rows are mostly empty
    (several staged chunks per row)."""
    if case == "config1":
        A = B = synth.config(1)
    elif case == "band":
        A = B = synth.banded(20000, 3, seed=2)
    elif case == "random_dup":
        A = synth.random_sparse(400, 300, 0.02, 7, duplicates=True, empty_rows=True, sort_rows=False)
        B = synth.random_sparse(300, 500, 0.01, 8, duplicates=True, empty_rows=True)
    else:
        from synth import CSR
        A = synth.random_sparse(200, 3000, 0.03, 9, duplicates=True)     # ~90 entries per row
        Bf = synth.random_sparse(3000, 400, 0.004, 10)
        keep = np.zeros(3000, dtype=bool)
        keep[::40] = True                                               # most B rows empty
        lens = np.diff(Bf.row_ptr) * keep
        rp = np.zeros(3001, np.int64)
        np.cumsum(lens, out=rp[1:])
        sel = np.repeat(keep, np.diff(Bf.row_ptr))
        B = CSR(3000, 400, rp, Bf.col[sel], Bf.val[sel])
    for kw in (None, opts(flags=4096)):  # expand-sort-compact (default), and hash tables
        rp, col, val, st = gpu_product(A, B, kw)
        compare_full(A, B, rp, col, val, threads=8)
