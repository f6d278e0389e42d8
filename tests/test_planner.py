"""Planner pins (host only): the chunk/level rule reproduces every "Num. Chunks" cell of the
gMAGNUS page, section IV, Tables V and VI, with the chunk width and per-level maximum the
tables imply (H200: W = 8192, 64 chunks per level; PVC: W = 4096, 32 per level); Eq. (4)
and Eq. (7) closed forms; rejection of malformed overrides."""
import os

import pytest

import sparse_gemm_irregular_gb300 as sg

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "gmagnus_chunk_tables.txt")


def _fmt(p):
    v = [str(p.v_chunks[i]) for i in range(p.levels)]
    return str(p.chunks_required) if p.levels == 1 else "%d: %s" % (p.chunks_required, ", ".join(v))


def _rows():
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        name, cm, pvc, h200 = [x.strip() for x in line.split("|")]
        yield name, int(cm), pvc, h200


@pytest.mark.parametrize("name,cm,pvc,h200", list(_rows()))
def test_tables_v_vi(name, cm, pvc, h200):
    s_lm = 232448
    p = sg.spgemm_plan_params(cm, s_lm, sg.options(chunk_width=8192, chunks_max=64))
    assert _fmt(p) == h200, name
    if pvc != "-":
        p = sg.spgemm_plan_params(cm, s_lm, sg.options(chunk_width=4096, chunks_max=32))
        assert _fmt(p) == pvc, name


def test_golden_has_all_cells():
    rows = list(_rows())
    assert len(rows) == 26
    assert sum(1 for r in rows if r[2] != "-") + len(rows) == 51


def test_eq4_tau_and_dense_width():
    for s_lm in (65536, 98304, 131072, 225280):
        p = sg.spgemm_plan_params(1 << 20, s_lm)
        assert p.tau == s_lm // 24                       # alpha = 2, s_col = 4, s_val = 8
        assert p.dense_numeric == (s_lm * 8) // 65       # s_LM / (8 + 1/8)
        w = p.chunk_width
        assert w & (w - 1) == 0 and w <= p.dense_numeric < 2 * w


@pytest.mark.parametrize("req,mx", [(2, 2), (64, 8), (128, 8), (1 << 12, 16), (1 << 13, 4)])
def test_eq7_levels(req, mx):
    W = 64
    p = sg.spgemm_plan_params(req * W, 232448, sg.options(chunk_width=W, chunks_max=mx))
    assert p.chunks_required == req
    lr, lm = req.bit_length() - 1, mx.bit_length() - 1
    expect = 1 if req <= mx else -(-lr // lm)
    assert p.levels == expect
    prod = 1
    for i in range(p.levels):
        prod *= p.v_chunks[i]
    assert prod == req                                   # the levels multiply to the requirement
    assert all(p.v_chunks[i] == mx for i in range(p.levels - 1))


def test_group_rows():
    p = sg.spgemm_plan_params(1 << 18, 232448, sg.options(tau=1000))
    assert p.group_rows == -(-(p.group_elems_ms - 1) // 1000) + 1


@pytest.mark.parametrize("kw", [dict(chunk_width=3000), dict(chunks_max=6), dict(chunks_max=1),
                                dict(tau=-1), dict(chunk_width=1 << 20)])
def test_rejects_bad_overrides(kw):
    with pytest.raises(sg.SpgemmError):
        sg.spgemm_plan_params(1 << 16, 232448, sg.options(**kw))
