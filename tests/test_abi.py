"""The C ABI on the host: the library loads, exports every function include/spgemm.h declares,
and rejects malformed calls before touching a GPU."""
import ctypes
import os
import re

import pytest

import sparse_gemm_irregular_gb300 as sg
from sparse_gemm_irregular_gb300 import binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "spgemm.h")


def declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spgemm_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol():
    lib = ctypes.CDLL(binding.LIB_PATH)
    names = declared()
    assert "spgemm_create" in names and "spgemm_numeric_rows" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(binding.EXPORTS)


def test_strerror_and_codes():
    assert sg.spgemm_strerror(0) == "ok"
    for code in binding.ERRORS:
        assert sg.spgemm_strerror(code) not in ("ok", "unknown status")


def test_create_rejects_shape_mismatch_without_gpu():
    lib = sg.load()
    A = binding.spgemm_csr(4, 5, 0, 1, 0, 0)   # fake non-null row_ptr; never dereferenced
    B = binding.spgemm_csr(6, 3, 0, 1, 0, 0)   # B.rows != A.cols
    h = ctypes.c_void_p()
    rc = lib.spgemm_create(ctypes.byref(h), 4, 5, 3, ctypes.byref(A), ctypes.byref(B), None)
    assert rc == -1 and not h.value
    rc = lib.spgemm_create(ctypes.byref(h), -1, 5, 3, ctypes.byref(A), ctypes.byref(B), None)
    assert rc == -1
    big = binding.spgemm_csr(5, 1 << 32, 0, 1, 0, 0)
    B2 = binding.spgemm_csr(1 << 32, 3, 0, 1, 0, 0)
    rc = lib.spgemm_create(ctypes.byref(h), 5, 1 << 32, 3, ctypes.byref(big), ctypes.byref(B2), None)
    assert rc == -5
    assert lib.spgemm_destroy(None) == 0


def test_null_handle_calls():
    lib = sg.load()
    nnz = ctypes.c_int64()
    assert lib.spgemm_symbolic(None, None, ctypes.byref(nnz)) == -1
    assert lib.spgemm_numeric(None, None, None) == -1
    assert lib.spgemm_numeric_rows(None, 0, 1, None, None) == -1


def test_struct_layouts_match_the_header(tmp_path):
    """The ctypes structures of the binding against sizeof/offsetof of the C header (gcc)."""
    import shutil
    import subprocess
    if not shutil.which("gcc"):
        pytest.skip("no host C compiler")
    structs = {"spgemm_csr": binding.spgemm_csr, "spgemm_options": binding.spgemm_options,
               "spgemm_plan": binding.spgemm_plan, "spgemm_stats": binding.spgemm_stats}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "spgemm.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append('printf("%s %%zu\\n", sizeof(%s));' % (name, name))
        for fname, _ in cls._fields_:
            lines.append('printf("%s.%s %%zu\\n", offsetof(%s, %s));' % (name, fname, name, fname))
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)])
    got = dict(l.rsplit(" ", 1) for l in subprocess.check_output([str(exe)], text=True).splitlines())
    for name, cls in structs.items():
        assert int(got[name]) == ctypes.sizeof(cls), name
        for fname, _ in cls._fields_:
            assert int(got["%s.%s" % (name, fname)]) == getattr(cls, fname).offset, (name, fname)


def test_new_entry_points_reject_bad_arguments_without_gpu():
    lib = sg.load()
    A = binding.spgemm_csr(4, 5, 0, 1, 0, 0)
    B = binding.spgemm_csr(5, 3, 0, 1, 0, 0)
    Bbad = binding.spgemm_csr(6, 3, 0, 1, 0, 0)
    cap = ctypes.c_void_p(1)
    assert lib.spgemm_hll_estimate(ctypes.byref(A), ctypes.byref(B), 48, ctypes.c_double(1.5), cap, None) == -1
    assert lib.spgemm_hll_estimate(ctypes.byref(A), ctypes.byref(B), 64, ctypes.c_double(0.0), cap, None) == -1
    assert lib.spgemm_hll_estimate(ctypes.byref(A), ctypes.byref(Bbad), 64, ctypes.c_double(1.5), cap, None) == -1
    assert lib.spgemm_hll_estimate(None, ctypes.byref(B), 64, ctypes.c_double(1.5), cap, None) == -1
    nnz = ctypes.c_int64()
    C = binding.spgemm_csr(4, 3, 0, 1, 0, 0)
    assert lib.spgemm_mcl_prune_symbolic(ctypes.byref(C), ctypes.c_double(-1.0), cap, cap, ctypes.byref(nnz),
                                         None) == -1
    assert lib.spgemm_mcl_prune_symbolic(ctypes.byref(C), ctypes.c_double(0.002), cap, None, ctypes.byref(nnz),
                                         None) == -1
    assert lib.spgemm_mcl_prune_numeric(None, ctypes.c_double(0.002), cap, cap, cap, cap, None) == -1
    h = ctypes.c_void_p()
    for kw in (dict(workflow=4), dict(workflow=-1), dict(hll_registers=16), dict(hll_coef=-0.5)):
        o = sg.options(**kw)
        rc = lib.spgemm_create_ex(ctypes.byref(h), 4, 5, 3, ctypes.byref(A), ctypes.byref(B), None, ctypes.byref(o))
        assert rc == -1 and not h.value, kw
