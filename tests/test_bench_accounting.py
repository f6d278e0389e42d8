"""The bench's byte accounting, on CPU: the algorithmic bytes per heavy product of each plan, the
compulsory bytes of a product worked by hand, and the DRAM traffic read from a committed ncu
summary only while the kernel's source is the one that was captured."""
import hashlib
import os
import sys
from types import SimpleNamespace

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _bench():
    import bench
    return bench


def _stats(resident, gen, e=1000, dense_elems=600, dense_nnz=250):
    return SimpleNamespace(ip_heavy=e, resident=resident, gen_symbolic=gen, dense_elems=dense_elems,
                           dense_nnz=dense_nnz)


def test_outer_product_bytes_per_plan():
    kb = _bench().kernel_bytes
    # one expansion with values (resident C^_reord, or chunks counted from generated products)
    assert kb("outer_product", _stats(1, 0)) == 12 * 1000
    assert kb("outer_product", _stats(0, 1)) == 12 * 1000
    # columns in the symbolic phase, then columns and values in the numeric one
    assert kb("outer_product", _stats(0, 0)) == 16 * 1000
    # the separate multisplit reads and writes C^ once, or twice when recomputed
    assert kb("multisplit", _stats(1, 0)) == 24 * 1000
    assert kb("multisplit", _stats(0, 0)) == 32 * 1000
    assert kb("chunk_symbolic", _stats(1, 0)) == 4 * 1000
    # dense chunks: their elements read, their entries of C written
    assert kb("chunk_dense", _stats(1, 0)) == 12 * 600 + 12 * 250
    assert kb("no_such_kernel", _stats(1, 0)) is None


def test_compulsory_bytes_worked_example():
    cb = _bench().compulsory_bytes
    # A 2x3 with entries in columns 0 and 2; B 3x2 with rows of 1, 2 and 3 entries: A touches
    # rows 0 and 2 of B (1 + 3 entries); C has 3 entries
    A = SimpleNamespace(rows=2, nnz=3, col=np.array([0, 2, 2]), row_ptr=np.array([0, 2, 3]))
    B = SimpleNamespace(rows=3, nnz=6, col=np.array([0, 0, 1, 0, 1, 1]), row_ptr=np.array([0, 1, 3, 6]))
    want = (3 * 8 + 12 * 3) + (4 * 8 + 12 * 4) + (3 * 8 + 12 * 3)
    assert cb(A, B, 3) == want


def _traffic_tree(tmp_path, body, src_text):
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "sparse_gemm_irregular_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k_demo.cu").write_text(src_text)
    sha = hashlib.sha1(src_text.encode()).hexdigest()[:12]
    (tmp_path / "profiles" / "traffic_demo_w.md").write_text(body.format(sha=sha))
    return csrc / "k_demo.cu"


def test_measured_traffic_follows_the_source(tmp_path, monkeypatch):
    bench = _bench()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = _traffic_tree(tmp_path, "# summary\n\n    traffic k_demo source=k_demo.cu sha1={sha} bytes=123456\n",
                        "kernel source\n")
    assert bench.measured_traffic("k_demo", "demo_w") == 123456
    assert bench.measured_traffic("k_other", "demo_w") is None
    assert bench.measured_traffic("k_demo", "missing_w") is None
    src.write_text("kernel source, changed\n")   # counters no longer describe this kernel
    assert bench.measured_traffic("k_demo", "demo_w") is None
    src.unlink()
    assert bench.measured_traffic("k_demo", "demo_w") is None


@pytest.mark.parametrize("name", ["traffic_rmat_s18.md", "traffic_rmat_s21_ef32.md"])
def test_committed_traffic_lines_name_existing_sources(name):
    path = os.path.join(ROOT, "profiles", name)
    # the lines bench.measured_traffic reads: traffic <kernel> source=... sha1=... bytes=...
    lines = [p for p in (ln.split() for ln in open(path))
             if len(p) == 5 and p[0] == "traffic" and p[2].startswith("source=")]
    assert lines, "no machine-readable traffic line in " + name
    for parts in lines:
        kv = dict(x.split("=", 1) for x in parts[2:])
        assert set(kv) == {"source", "sha1", "bytes"}
        assert os.path.exists(os.path.join(ROOT, "sparse_gemm_irregular_gb300", "csrc", kv["source"]))
        assert len(kv["sha1"]) == 12 and int(kv["bytes"]) > 0
