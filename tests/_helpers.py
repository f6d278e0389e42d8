"""Shared helpers of the GPU parity tests: run the library through the C ABI, compare with the
oracle.  Bar: row_ptr and col_idx bit-exact; every value within 1e-12 of the oracle's sum of
|products| for that entry (the tolerance stated for the values, read relative to the absolute
sum so that entries that cancel towards zero stay well-posed)."""
import numpy as np

import oracle

RTOL = 1e-12


def gpu_product(A, B, opts=None, check_stats=True):
    import torch
    import sparse_gemm_irregular_gb300 as sg
    dA = sg.DeviceCSR.from_host(A)
    dB = dA if B is A else sg.DeviceCSR.from_host(B)
    p = sg.Product(dA, dB, opts=opts)
    try:
        rp, nnz = p.symbolic()
        col, val = p.numeric()
        torch.cuda.synchronize()
        st = p.stats()
    finally:
        p.close()
    return rp.cpu().numpy(), col.cpu().numpy()[:nnz], val.cpu().numpy()[:nnz], st


def compare_full(A, B, rp, col, val, threads=8):
    orp, ocol, oval, oabs = oracle.spgemm_rows(A, B, np.arange(A.rows), threads=threads)
    assert rp.shape == orp.shape
    bad = np.nonzero(rp != orp)[0]
    assert len(bad) == 0, "row_ptr differs first at %d: gpu %d oracle %d" % (bad[0], rp[bad[0]], orp[bad[0]])
    assert np.array_equal(col, ocol), "col_idx differs first at %d" % np.nonzero(col != ocol)[0][0]
    err = np.abs(val - oval)
    ok = err <= RTOL * oabs
    assert ok.all(), "value differs at %d: gpu %r oracle %r abs %r" % (
        np.nonzero(~ok)[0][0], val[~ok][0], oval[~ok][0], oabs[~ok][0])
    return float((err / np.where(oabs > 0, oabs, 1)).max()) if len(err) else 0.0


def compare_rows(A, B, rp, col, val, rows, threads=8):
    """Compare a sample of rows of the GPU result (full row_ptr, col, val) with the oracle."""
    rows = np.ascontiguousarray(np.sort(rows), np.int64)
    orp, ocol, oval, oabs = oracle.spgemm_rows(A, B, rows, threads=threads)
    worst = 0.0
    for j, i in enumerate(rows):
        a, b = int(rp[i]), int(rp[i + 1])
        oa, ob = int(orp[j]), int(orp[j + 1])
        assert b - a == ob - oa, "row %d: nnz gpu %d oracle %d" % (i, b - a, ob - oa)
        assert np.array_equal(col[a:b], ocol[oa:ob]), "row %d: columns differ" % i
        err = np.abs(val[a:b] - oval[oa:ob])
        assert np.all(err <= RTOL * oabs[oa:ob]), "row %d: values differ" % i
        if b > a:
            worst = max(worst, float((err / np.where(oabs[oa:ob] > 0, oabs[oa:ob], 1)).max()))
    return worst


def invariants(A, B, rp, col, val):
    """Properties that hold at any size: nnz per row <= IP per row, sorted unique columns,
    row sums of C equal A times the row sums of B, and C x = A (B x) (Freivalds)."""
    ip = oracle.row_ip(A, B)
    nnz = np.diff(rp)
    assert rp[0] == 0 and np.all(nnz >= 0) and np.all(nnz <= ip)
    assert np.all((nnz > 0) == (ip > 0))
    if len(col):
        rows = np.repeat(np.arange(A.rows), nnz)
        d = np.diff(col.astype(np.int64))
        same_row = rows[1:] == rows[:-1]
        assert np.all(d[same_row] > 0), "columns not strictly increasing inside a row"
        assert col.min() >= 0 and col.max() < B.cols
    x = np.random.default_rng(0).random(B.cols)
    bx = np.zeros(B.rows)
    np.add.at(bx, np.repeat(np.arange(B.rows), np.diff(B.row_ptr)), B.val * x[B.col])
    abx = np.zeros(A.rows)
    np.add.at(abx, np.repeat(np.arange(A.rows), np.diff(A.row_ptr)), A.val * bx[A.col])
    cx = np.zeros(A.rows)
    np.add.at(cx, np.repeat(np.arange(A.rows), nnz), val * x[col])
    # tolerance from |A| |B| |x|
    bax = np.zeros(B.rows)
    np.add.at(bax, np.repeat(np.arange(B.rows), np.diff(B.row_ptr)), np.abs(B.val) * x[B.col])
    scale = np.zeros(A.rows)
    np.add.at(scale, np.repeat(np.arange(A.rows), np.diff(A.row_ptr)), np.abs(A.val) * bax[A.col])
    assert np.all(np.abs(cx - abx) <= 1e-11 * scale + 1e-300)


def gpu_product_device(A, B, opts=None):
    """Run the product and keep C on the device: (Product, row_ptr, col, val) as torch tensors."""
    import torch
    import sparse_gemm_irregular_gb300 as sg
    dA = sg.DeviceCSR.from_host(A)
    dB = dA if B is A else sg.DeviceCSR.from_host(B)
    p = sg.Product(dA, dB, opts=opts)
    rp, nnz = p.symbolic()
    col, val = p.numeric()
    torch.cuda.synchronize()
    return p, rp, col, val


def device_invariants(A, B, rp, col, val, chunk=1 << 28):
    """Invariants of C = A B checked with torch on the device, in element chunks (C may be far
    larger than host memory): nnz per row <= IP per row, strictly increasing columns inside
    every row, C x = A (B x) for a random x.  Returns (row sums, column sums) of C."""
    import torch
    dev = rp.device
    m, n = A.rows, B.cols
    ip = torch.from_numpy(oracle.row_ip(A, B)).to(dev)
    nnz_row = rp[1:] - rp[:-1]
    assert int(rp[0]) == 0 and bool((nnz_row >= 0).all()) and bool((nnz_row <= ip).all())
    assert bool(((nnz_row > 0) == (ip > 0)).all())
    x = torch.from_numpy(np.random.default_rng(0).random(n)).to(dev)
    rowsum = torch.zeros(m, dtype=torch.float64, device=dev)
    colsum = torch.zeros(n, dtype=torch.float64, device=dev)
    cx = torch.zeros(m, dtype=torch.float64, device=dev)
    total = int(rp[-1])
    for e0 in range(0, total, chunk):
        e1 = min(total, e0 + chunk)
        pos = torch.arange(e0, e1, device=dev, dtype=torch.int64)
        rows = torch.searchsorted(rp, pos, right=True) - 1
        c = col[e0:e1].long()
        v = val[e0:e1]
        assert bool((c >= 0).all()) and bool((c < n).all())
        same = rows[1:] == rows[:-1]
        assert bool((c[1:] > c[:-1])[same].all()), "columns not increasing inside a row"
        if e0 > 0:
            r_prev = int(torch.searchsorted(rp, torch.tensor([e0 - 1], device=dev), right=True)[0]) - 1
            if r_prev == int(rows[0]):
                assert int(col[e0 - 1]) < int(c[0])
        rowsum.index_add_(0, rows, v)
        colsum.index_add_(0, c, v)
        cx.index_add_(0, rows, v * x[c])
        del pos, rows, c, v, same
    # reference A (B x) and its absolute scale on the host
    xh = x.cpu().numpy()
    def spmv(M, y, absolute=False):
        out = np.zeros(M.rows)
        vals = np.abs(M.val) if absolute else M.val
        np.add.at(out, np.repeat(np.arange(M.rows), np.diff(M.row_ptr)), vals * y[M.col])
        return out
    bx = spmv(B, xh)
    abx = spmv(A, bx)
    scale = spmv(A, spmv(B, np.abs(xh), True), True)
    assert np.all(np.abs(cx.cpu().numpy() - abx) <= 1e-11 * scale + 1e-300)
    return rowsum, colsum


def device_rows(rp, col, val, rows):
    """Gather the listed rows of a device CSR to the host: (row_ptr over the list, col, val)."""
    import torch
    rph = rp.cpu().numpy()
    out_rp = [0]
    cols, vals = [], []
    for i in rows:
        a, b = int(rph[i]), int(rph[i + 1])
        cols.append(col[a:b].cpu().numpy())
        vals.append(val[a:b].cpu().numpy())
        out_rp.append(out_rp[-1] + b - a)
    return (np.array(out_rp, np.int64), np.concatenate(cols) if cols else np.zeros(0, np.int32),
            np.concatenate(vals) if vals else np.zeros(0))


def release_device_memory():
    import torch
    import sparse_gemm_irregular_gb300 as sg
    torch.cuda.synchronize()
    sg.spgemm_release_memory()
    torch.cuda.empty_cache()


def compare_sampled_device(A, B, rp, col, val, rows, threads=16):
    rows = np.ascontiguousarray(np.sort(np.unique(rows)), np.int64)
    grp, gcol, gval = device_rows(rp, col, val, rows)
    orp, ocol, oval, oabs = oracle.spgemm_rows(A, B, rows, threads=threads)
    assert np.array_equal(grp, orp), "row sizes differ on the sample"
    assert np.array_equal(gcol, ocol), "columns differ on the sample"
    assert np.all(np.abs(gval - oval) <= RTOL * oabs), "values differ on the sample"
