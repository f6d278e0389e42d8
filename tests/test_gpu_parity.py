"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element by element.

Small and medium inputs are compared in full (the full-size workloads are compared in
test_gpu_fullsize.py); the direct split of level 0 is also checked at full size on a sample of
rows (all the heaviest rows plus a seeded uniform sample) and through invariants that hold at
any size.  Planner overrides force the rare paths on small inputs:
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
    # heavy rows by the long-row hash (shared table spilling to a global one): small shared tables
    # would not spill on these sizes, so every row is heavy and long enough
    dict(flags=32768 | 1, tau=16),
    dict(flags=32768, tau=64, heavy_batch_elems=700),
    # recomputed one-level plans count their chunks from generated products by default; this
    # keeps the column expansion in the symbolic phase
    dict(flags=65536 | 16, tau=16, chunk_width=64, chunks_max=16, heavy_batch_elems=700),
    # the two numeric hash bins by a warp or block per chunk instead of persistent groups
    dict(flags=131072, tau=16, chunk_width=64, chunks_max=16),
    dict(flags=131072 | 16, tau=16, chunk_width=64, chunks_max=16, heavy_batch_elems=700),
    # one-level plans through the separate outer product and multisplit pass
    dict(flags=16384 | 1, tau=64, chunk_width=64, chunks_max=8),
    dict(flags=16384, tau=16, chunk_width=64, chunks_max=16, heavy_batch_elems=700),
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


@pytest.mark.parametrize("flags", [0, 64, 128, 256, 512, 1024, 4096, 8192, 16384, 32768, 131072])
def test_rmat_small_full(gpu_lib, flags):
    """R-MAT scale 14, edge factor 16: heavy rows above the default tau, several chunks per
    row (dense chunks among them), thousands of light rows in every ladder bin -- compared in
    full (multisplit path, plain shared atomics in the multisplit, dense chunks in L2, direct
    split, bulk-copy staged multisplit, per-product level-0 histogram, short hash rows in
    shared hash tables instead of expand-sort-compact, heavy chunks generated from the
    column-split B, the separate multisplit pass of a one-level plan, heavy rows by the long-row
    hash)."""
    A = synth.rmat(14, 16, seed=5)
    rp, col, val, st = gpu_product(A, A, opts(flags=flags) if flags else None)
    assert st.rows_heavy > 0 and st.rows_light > 0
    assert st.dense_elems > 0 or flags & 32768
    assert st.long_rows == (1 if flags & 32768 else 0)
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


# the default (level 0 split inside the outer product) and generating paths are compared in full
# at this size (test_gpu_fullsize.py); here the separate multisplit pass, on sampled rows and
# invariants
@pytest.mark.parametrize("flags", [16384])
def test_config3_full_size_sampled(gpu_lib, flags):
    A = synth.config(3)
    p, rp, col, val = gpu_product_device(A, A, opts(flags=flags) if flags else None)
    st = p.stats()
    assert st.rows_heavy > 0 and st.resident == 1
    rowsum, _ = device_invariants(A, A, rp, col, val)
    compare_sampled_device(A, A, rp, col, val, sample_rows(A, A))
    p.close()
    del rp, col, val
    release_device_memory()


@pytest.mark.parametrize("flags", [16384])
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
                                         ("rmat", 1), ("fused", 3000), ("fused_batches", 3000), ("long", 3000)])
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
    elif case == "long":
        A, B, kw = synth.rmat(13, 16, seed=8), None, dict(flags=32768, tau=512)
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


def _csr(rows, cols, entries):
    """CSR from a list of (row, col, value) in the given order (duplicates kept)."""
    from synth import CSR
    entries = sorted(entries, key=lambda t: t[0])  # stable: keeps the order inside each row
    rp = np.zeros(rows + 1, np.int64)
    for r, _, _ in entries:
        rp[r + 1] += 1
    return CSR(rows, cols, np.cumsum(rp), np.array([c for _, c, _ in entries], np.int32),
               np.array([v for _, _, v in entries], np.float64))


@pytest.mark.parametrize("kw", [None, dict(flags=1, tau=1, chunk_width=64, chunks_max=4),
                                dict(flags=8192 | 1, tau=1, chunk_width=64, chunks_max=4)])
def test_exact_cancellation_kept(gpu_lib, kw):
    """An entry whose products sum to exactly 0.0 stays in C with the value 0.0 (the symbolic
    phase fixes the structure before any value exists): A = [1 1], B = [2; -2], then a seeded
    product where every entry of half the rows cancels, on the light path and on both heavy
    paths."""
    A = _csr(1, 2, [(0, 0, 1.0), (0, 1, 1.0)])
    B = _csr(2, 1, [(0, 0, 2.0), (1, 0, -2.0)])
    rp, col, val, _ = gpu_product(A, B, opts(**kw) if kw else None)
    assert list(rp) == [0, 1] and list(col) == [0] and val[0] == 0.0
    # larger: rows 2k and 2k+1 of B are equal up to the sign and own columns 4k .. 4k+3 alone;
    # row i of A uses both rows of three pairs with the same weight when i is even (every column
    # then receives exactly +t and -t: zero in any order), different weights when odd
    vals = synth.uniform(31, 2, 0, 256, 0.5, 2.0)
    ent = []
    for k in range(64):
        for t in range(4):
            ent.append((2 * k, 4 * k + t, float(vals[4 * k + t])))
            ent.append((2 * k + 1, 4 * k + t, -float(vals[4 * k + t])))
    B2 = _csr(128, 300, ent)
    aent = []
    for i in range(200):
        for j in range(3):
            k = (7 * i + 13 * j) % 64
            w = 0.5 + j
            aent.append((i, 2 * k, w))
            aent.append((i, 2 * k + 1, w if i % 2 == 0 else 2 * w))
    A2 = _csr(200, 128, aent)
    rp, col, val, _ = gpu_product(A2, B2, opts(**kw) if kw else None)
    compare_full(A2, B2, rp, col, val)
    even = np.concatenate([np.arange(rp[i], rp[i + 1]) for i in range(0, 200, 2)])
    assert len(even) > 0 and np.all(val[even] == 0.0)  # present, exactly zero


def test_rows_at_tau(gpu_lib):
    """Rows with exactly tau intermediate products stay light, tau + 1 go heavy (gMAGNUS page,
    Algorithm 3, ThreshPartition: heavy means more than tau)."""
    tau = 64
    B = synth.random_sparse(40, 2000, 0.004, 41)            # rows of about 8 entries
    lens = np.diff(B.row_ptr)
    rng = np.random.default_rng(5)
    ent = []
    want = []
    for i in range(120):
        target = tau + (i % 3) - 1                            # tau - 1, tau, tau + 1
        s, row = 0, []
        while s < target:
            k = int(rng.integers(0, 40))
            if lens[k] == 0 or s + lens[k] > target:
                k = next((kk for kk in range(40) if 0 < lens[kk] <= target - s), None)
                if k is None:
                    break
            row.append(k)
            s += lens[k]
        if s != target:
            continue
        want.append(s)
        ent += [(len(want) - 1, k, 1.0 + 0.1 * j) for j, k in enumerate(row)]
    A = _csr(len(want), 40, ent)
    ip = oracle.row_ip(A, B)
    assert np.array_equal(ip, want) and {tau - 1, tau, tau + 1} <= set(ip.tolist())
    for flags in (0, 8192):
        rp, col, val, st = gpu_product(A, B, opts(tau=tau, chunk_width=256, flags=flags))
        assert st.rows_heavy == int((ip > tau).sum())
        compare_full(A, B, rp, col, val)


@pytest.mark.parametrize("flags", [0, 131072, 8192])
def test_chunks_at_hash_group_switch(gpu_lib, flags):
    """Final chunks of 256 elements (the largest on a warp group), 257 (the smallest on a block
    group), 66 with 33 distinct columns (just past a 64-slot table), 289, 513 and 770 elements
    (table sizes 1024 and 2048 of the block groups); by the persistent groups (default), one warp
    or block per chunk, and the generated chunks.  Chunk width 2048, every row heavy."""
    W = 2048
    ent_b = [(0, 3 * c, 1.0 + c / 512) for c in range(256)]               # 256 columns in chunk 0
    ent_b += [(1, W + 2 * c, 0.5 + c / 1024) for c in range(257)]         # 257 columns in chunk 1
    ent_b += [(2, 5 * c, -1.0 + c / 64) for c in range(33)]               # 33 columns in chunk 0
    ent_b += [(3, W + 3 * c, 0.25 + c / 2048) for c in range(513)]        # 513 columns in chunk 1
    B = _csr(4, 2 * W, ent_b)
    A = _csr(4, 4, [(0, 0, 1.5), (0, 1, -0.5),                # chunks of 256 and 257 elements
                    (1, 2, 1.0), (1, 2, 3.0), (1, 3, 0.75),   # 66 elements on 33 columns; 513
                    (2, 0, 2.0), (2, 2, -1.25),               # 289 elements, shared columns
                    (3, 1, 0.5), (3, 3, 1.5)])                # 770 elements
    rp, col, val, st = gpu_product(A, B, opts(tau=32, chunk_width=W, flags=flags))
    assert st.rows_heavy == 4
    compare_full(A, B, rp, col, val)


@pytest.mark.parametrize("flags", [0, 8192])
def test_chunks_at_dense_switch(gpu_lib, flags):
    """Final chunks of exactly 1024 elements take a hash accumulator, 1025 the dense one (the
    hash/dense switch of the last level); chunk width 2048, one heavy row per case."""
    W = 2048
    ent_b = [(0, c, 1.0 + c / 4096) for c in range(1024)]                 # 1024 columns in chunk 0
    ent_b += [(1, W + c, 0.5 + c / 8192) for c in range(1025)]            # 1025 columns in chunk 1
    ent_b += [(2, c * 2, 2.0) for c in range(512)]                        # 512 columns in chunk 0
    B = _csr(3, 2 * W, ent_b)
    A = _csr(3, 3, [(0, 0, 1.5), (0, 1, -0.5),                            # chunks of 1024 and 1025
                    (1, 2, 1.0), (1, 2, 3.0), (1, 0, 0.25),               # 1024 + 1024 duplicates-heavy
                    (2, 1, 2.0)])                                         # one chunk of 1025
    rp, col, val, st = gpu_product(A, B, opts(tau=1000, chunk_width=W, flags=flags))
    assert st.rows_heavy == 3 and st.chunks_dense >= 2
    compare_full(A, B, rp, col, val)
