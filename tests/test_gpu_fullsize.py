"""Full-size parity on the three large workloads, through the C ABI, against the oracle.

R-MAT scale 18 (2.9e9 products) and the Markov-clustering expansion (R-MAT scale 20 + I,
column-stochastic, 2.1e10 products) are compared in full: every row of C, streamed in row
windows (spgemm_row_windows + spgemm_numeric_rows into one reused device buffer), each window
copied to the host in blocks and compared with the oracle's rows (dense accumulator, all host
cores).  R-MAT scale 21 (1.9e11 products, C of 6.7e10 entries: larger than the device and the
host) is compared on its full row_ptr (the oracle's row sizes of every row), on every row of
the 1000 heaviest and 10,000 seeded uniform rows (values included), and on properties of every
entry of every window: columns strictly increasing inside each row, and C x = A (B x) row by
row.  Both heavy-row paths are covered: the expanded one (outer product + multisplit, the
default) and the generating one (SPGEMM_FLAG_FUSED)."""
import os

import numpy as np
import pytest

import oracle
import synth
from _helpers import RTOL, release_device_memory

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 1
HOST_BLOCK = 1 << 27        # entries of C per host comparison block
WINDOW = 1 << 29            # entries of C per numeric window (windows hold whole heavy batches)

_cache = {}


def workload(cid):
    if cid not in _cache:
        _cache.clear()
        _cache[cid] = synth.config(cid)
    return _cache[cid]


def _spmv(M, y, absolute=False):
    v = np.abs(M.val) if absolute else M.val
    return np.bincount(np.repeat(np.arange(M.rows), np.diff(M.row_ptr)), weights=v * y[M.col], minlength=M.rows)


def _check_window_device(col, val, lrp_dev, x_dev):
    """Columns strictly increasing inside every row of the window; returns C x for its rows."""
    import torch
    nrows = lrp_dev.numel() - 1
    total = int(lrp_dev[-1])
    cx = torch.zeros(nrows, dtype=torch.float64, device=col.device)
    for e0 in range(0, total, 1 << 28):
        e1 = min(total, e0 + (1 << 28))
        pos = torch.arange(e0, e1, device=col.device, dtype=torch.int64)
        rows = torch.searchsorted(lrp_dev, pos, right=True) - 1
        c = col[e0:e1].long()
        same = rows[1:] == rows[:-1]
        assert bool((c[1:] > c[:-1])[same].all()), "columns not increasing inside a row"
        if e0 > 0 and int(rows[0]) == int(torch.searchsorted(lrp_dev, torch.tensor([e0 - 1], device=col.device),
                                                             right=True)[0]) - 1:
            assert int(col[e0 - 1]) < int(c[0])
        cx.index_add_(0, rows, val[e0:e1] * x_dev[c])
        del pos, rows, c, same
    return cx.cpu().numpy()


def stream_parity(A, prods, rp_host, sample=None):
    """Numeric phase of every product handle in `prods` (the same product by different paths),
    window by window into reused device buffers.  Every window of every product is checked on
    the device (order, Freivalds); its rows (all, or only `sample`) are compared with the
    oracle, computed once for all the products.  Returns the number of rows compared."""
    import torch
    cuts, wmax = prods[0].row_windows(WINDOW)
    for q in prods[1:]:
        wmax = max(wmax, q.row_windows(WINDOW)[1])
    # the other paths may cut elsewhere; the largest window over these cuts bounds every buffer
    wmax = max(wmax, max(int(rp_host[b] - rp_host[a]) for a, b in zip(cuts[:-1], cuts[1:])))
    bufs = [(torch.empty(max(wmax, 1), dtype=torch.int32, device="cuda"),
             torch.empty(max(wmax, 1), dtype=torch.float64, device="cuda")) for _ in prods]
    x = synth.uniform(11, synth.STREAM_SAMPLE, 0, A.cols, 0.0, 1.0)
    x_dev = torch.from_numpy(x).cuda()
    bx, bax = _spmv(A, x), _spmv(A, x, True)
    compared = 0
    for rb, re in zip(cuts[:-1], cuts[1:]):
        lrp = rp_host[rb:re + 1] - rp_host[rb]
        lrp_dev = torch.from_numpy(lrp).cuda()
        a0, a1 = A.row_ptr[rb], A.row_ptr[re]
        arid = np.repeat(np.arange(re - rb), np.diff(A.row_ptr[rb:re + 1]))
        ref = np.bincount(arid, weights=A.val[a0:a1] * bx[A.col[a0:a1]], minlength=re - rb)
        scale = np.bincount(arid, weights=np.abs(A.val[a0:a1]) * bax[A.col[a0:a1]], minlength=re - rb)
        for q, (dcol, dval) in zip(prods, bufs):
            q.numeric_rows(rb, re, dcol, dval)
            torch.cuda.synchronize()
            cx = _check_window_device(dcol, dval, lrp_dev, x_dev)
            assert np.all(np.abs(cx - ref) <= 1e-11 * scale + 1e-300), "C x != A (B x) in rows %d..%d" % (rb, re)
        if sample is None:
            r = rb
            while r < re:
                r2 = int(np.searchsorted(rp_host, rp_host[r] + HOST_BLOCK, side="right")) - 1
                r2 = min(re, max(r2, r + 1))
                o0, o1 = int(rp_host[r] - rp_host[rb]), int(rp_host[r2] - rp_host[rb])
                orp, ocol, oval, oabs = oracle.spgemm_rows(A, A, np.arange(r, r2), threads=THREADS,
                                                           accumulator="dense")
                assert np.array_equal(orp, rp_host[r:r2 + 1] - rp_host[r]), "row sizes differ in %d..%d" % (r, r2)
                for dcol, dval in bufs:
                    c = dcol[o0:o1].cpu().numpy()
                    assert np.array_equal(c, ocol), "columns differ in rows %d..%d" % (r, r2)
                    del c
                    v = dval[o0:o1].cpu().numpy()
                    assert not (np.abs(v - oval) > RTOL * oabs).any(), "values differ in rows %d..%d" % (r, r2)
                    del v
                del orp, ocol, oval, oabs
                compared += r2 - r
                r = r2
        else:
            rows = sample[(sample >= rb) & (sample < re)]
            if len(rows) == 0:
                continue
            starts = torch.from_numpy(rp_host[rows] - rp_host[rb]).cuda()
            lens = torch.from_numpy(rp_host[rows + 1] - rp_host[rows]).cuda()
            idx = torch.repeat_interleave(starts, lens) + (
                torch.arange(int(lens.sum()), device="cuda") - torch.repeat_interleave(
                    torch.cumsum(lens, 0) - lens, lens))
            orp, ocol, oval, oabs = oracle.spgemm_rows(A, A, rows, threads=THREADS, accumulator="dense")
            assert np.array_equal(np.diff(orp), rp_host[rows + 1] - rp_host[rows])
            for dcol, dval in bufs:
                c = dcol[idx].cpu().numpy()
                v = dval[idx].cpu().numpy()
                assert np.array_equal(c, ocol), "columns differ on the sampled rows of %d..%d" % (rb, re)
                assert not (np.abs(v - oval) > RTOL * oabs).any(), "values differ on the sampled rows"
            compared += len(rows)
            del idx, starts, lens
    del bufs
    return compared


def products(A):
    """The same product by the default (expanded) and the generating heavy-row path."""
    import sparse_gemm_irregular_gb300 as sg
    dA = sg.DeviceCSR.from_host(A)
    prods, rp_host, nnz = [], None, None
    for flags in (0, sg.binding.FLAG_FUSED):
        p = sg.Product(dA, dA, opts=sg.options(flags=flags) if flags else None)
        rp, n = p.symbolic()
        rph = rp.cpu().numpy()
        del rp
        if rp_host is None:
            rp_host, nnz = rph, n
        assert np.array_equal(rph, rp_host) and n == nnz, "row_ptr differs between the paths"
        prods.append(p)
    return dA, prods, rp_host, nnz


def close(dA, prods):
    for p in prods:
        p.close()
    del dA
    release_device_memory()


@pytest.mark.parametrize("cid", [3, 5])
def test_full_parity_streamed(gpu_lib, cid):
    """Every row of C against the oracle (R-MAT scale 18; Markov-clustering expansion), by both
    heavy-row paths."""
    A = workload(cid)
    dA, prods, rp_host, nnz = products(A)
    try:
        st = [p.stats() for p in prods]
        assert st[0].rows_heavy > 0 and st[0].fused == 0 and st[1].fused == 1
        assert rp_host[0] == 0 and rp_host[-1] == nnz
        assert stream_parity(A, prods, rp_host) == A.rows
    finally:
        close(dA, prods)


def test_config4_rowptr_and_sampled_rows(gpu_lib):
    """R-MAT scale 21, edge factor 32, by both heavy-row paths: C.row_ptr of every row against
    the oracle's row sizes; the 1000 heaviest rows (the rows the heavy path handles, up to 4e7
    products each) and 10,000 seeded uniform rows against the oracle's values; order and
    C x = A (B x) on every entry."""
    A = workload(4)
    ip = oracle.row_ip(A, A)
    dA, prods, rp_host, nnz = products(A)
    try:
        st = [p.stats() for p in prods]
        assert st[0].rows_heavy > 0 and st[0].resident == 0 and st[1].fused == 1
        ref_nnz = oracle.row_nnz(A, A, threads=THREADS)
        assert np.array_equal(np.diff(rp_host), ref_nnz)
        assert rp_host[0] == 0 and rp_host[-1] == nnz
        top = np.argsort(ip, kind="stable")[-1000:]
        uni = (synth.draws(0, synth.STREAM_SAMPLE, 0, 10000) % np.uint64(A.rows)).astype(np.int64)
        sample = np.unique(np.concatenate([top, uni]))
        assert ip[sample].max() == ip.max() and ip[sample].max() > 2_000_000
        assert stream_parity(A, prods, rp_host, sample=sample) == len(sample)
    finally:
        close(dA, prods)
