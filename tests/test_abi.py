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
