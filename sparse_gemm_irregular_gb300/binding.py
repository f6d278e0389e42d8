"""ctypes binding of libspgemm_gb300.so (include/spgemm.h): argument marshalling only.

The functions keep the C names.  Matrices live in PyTorch device tensors (torch is used
for device memory and streams); every step of the product runs in the library's kernels.
There is no CPU fallback: ``load()`` raises if the library is missing.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libspgemm_gb300.so")

SPGEMM_OK = 0
ERRORS = {
    -1: "INVALID_ARG", -2: "INVALID_CSR", -3: "BAD_STATE", -4: "OUT_OF_MEMORY",
    -5: "OVERFLOW", -6: "DEVICE", -7: "CUDA",
}
ERRORS_BY_NAME = {v: k for k, v in ERRORS.items()}
FLAG_ALL_HEAVY = 1
FLAG_ALL_LIGHT = 2
FLAG_NO_DENSE_LIGHT = 4
FLAG_VALIDATE = 8
FLAG_RECOMPUTE = 16
FLAG_TIMING = 32
FLAG_NO_MATCH = 64
FLAG_DENSE_L2 = 128
FLAG_DIRECT_SPLIT = 256
FLAG_TMA_SPLIT = 512
FLAG_FUSED_HIST = 1024
FLAG_NO_GRAPH = 2048
FLAG_NO_ESC = 4096
FLAG_FUSED = 8192
FLAG_EXPAND_SPLIT = 16384
FLAG_LONG_ROWS = 32768
FLAG_NO_GEN_SYMBOLIC = 65536
FLAG_HASH_PER_CHUNK = 131072
WORKFLOW_SYMBOLIC, WORKFLOW_UPPER_BOUND, WORKFLOW_ESTIMATE, WORKFLOW_AUTO = 0, 1, 2, 3
PHASES = ["setup", "light_symbolic", "masked_csc", "outer_product", "histogram", "multisplit",
          "multisplit_bookkeeping", "chunk_symbolic", "chunk_offsets", "rowptr_scan",
          "light_numeric", "chunk_numeric", "chunk_dense"]
MAX_LEVELS = 8

_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_vp = ctypes.c_void_p


class spgemm_csr(ctypes.Structure):
    _fields_ = [("rows", _i64), ("cols", _i64), ("nnz", _i64), ("row_ptr", _vp),
                ("col_idx", _vp), ("vals", _vp)]


class spgemm_options(ctypes.Structure):
    _fields_ = [("tau", _i64), ("chunk_width", _i64), ("chunks_max", _i64),
                ("heavy_batch_elems", _i64), ("smem_bytes", _i64), ("flags", _i32),
                ("workflow", _i32), ("hll_registers", _i32), ("reserved", _i32), ("hll_coef", ctypes.c_double),
                ("workspace_limit", _i64), ("debug_hash_slots", _i32), ("debug_wait_spins", _i32)]


class spgemm_plan(ctypes.Structure):
    _fields_ = [("s_lm", _i64), ("tau", _i64), ("dense_numeric", _i64), ("chunk_width", _i64),
                ("chunks_required", _i64), ("chunks_max", _i64), ("levels", _i32),
                ("reserved", _i32), ("v_chunks", _i64 * MAX_LEVELS), ("group_elems_op", _i64),
                ("group_elems_ms", _i64), ("group_rows", _i64)]


class spgemm_stats(ctypes.Structure):
    _fields_ = [("m", _i64), ("k", _i64), ("n", _i64), ("ip_total", _i64), ("ip_heavy", _i64),
                ("rows_heavy", _i64), ("rows_light", _i64), ("rows_empty", _i64),
                ("rows_dense_light", _i64), ("c_nnz", _i64), ("heavy_batches", _i64),
                ("levels_run", _i64), ("final_chunks", _i64), ("chunks_dense", _i64),
                ("chat_bytes", _i64), ("c_nnz_heavy", _i64), ("dense_elems", _i64), ("dense_nnz", _i64),
                ("resident", _i32), ("numeric_graph", _i32), ("rows_overflow", _i64), ("workflow", _i32),
                ("hll_registers", _i32), ("fused", _i32), ("direct_split", _i32), ("long_rows", _i32),
                ("gen_symbolic", _i32)]


EXPORTS = {
    "spgemm_plan_params": (ctypes.c_int, [_i64, _i64, _vp, _vp]),
    "spgemm_create": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp]),
    "spgemm_create_ex": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "spgemm_symbolic": (ctypes.c_int, [_vp, _vp, _vp]),
    "spgemm_numeric": (ctypes.c_int, [_vp, _vp, _vp]),
    "spgemm_numeric_rows": (ctypes.c_int, [_vp, _i64, _i64, _vp, _vp]),
    "spgemm_numeric_host": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i64]),
    "spgemm_row_windows": (ctypes.c_int, [_vp, _i64, _vp, _i64, _vp, _vp]),
    "spgemm_get_stats": (ctypes.c_int, [_vp, _vp]),
    "spgemm_get_plan": (ctypes.c_int, [_vp, _vp]),
    "spgemm_get_phase_times": (ctypes.c_int, [_vp, _vp, _vp, _i32]),
    "spgemm_kernel_launches": (ctypes.c_longlong, []),
    "spgemm_symbolic_noalloc": (ctypes.c_int, [_i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp]),
    "spgemm_hll_estimate": (ctypes.c_int, [_vp, _vp, _i32, ctypes.c_double, _vp, _vp]),
    "spgemm_mcl_prune_symbolic": (ctypes.c_int, [_vp, ctypes.c_double, _vp, _vp, _vp, _vp]),
    "spgemm_mcl_prune_numeric": (ctypes.c_int, [_vp, ctypes.c_double, _vp, _vp, _vp, _vp, _vp]),
    "spgemm_release_memory": (ctypes.c_int, []),
    "spgemm_destroy": (ctypes.c_int, [_vp]),
    "spgemm_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "spgemm_last_error": (ctypes.c_char_p, []),
}

_lib = None


class SpgemmError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__("%s failed: %s (%s) %s" % (what, ERRORS.get(code, code),
                                                   _lib.spgemm_strerror(code).decode() if _lib else "",
                                                   _lib.spgemm_last_error().decode() if _lib else ""))


def load():
    """Load the built library (``__graft_entry__.build()`` / ``build.py`` makes it)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libspgemm_gb300.so is not built (%s); run sparse_gemm_irregular_gb300/build.py"
                               % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(rc: int, what: str):
    if rc != SPGEMM_OK:
        raise SpgemmError(rc, what)


# ---- thin wrappers with the C names --------------------------------------------------------
def spgemm_plan_params(c_cols: int, s_lm: int, options: spgemm_options | None = None) -> spgemm_plan:
    lib = load()
    out = spgemm_plan()
    _check(lib.spgemm_plan_params(c_cols, s_lm, ctypes.byref(options) if options else None,
                                  ctypes.byref(out)), "spgemm_plan_params")
    return out


def spgemm_create(m, k, n, A: spgemm_csr, B: spgemm_csr, stream: int = 0,
                  options: spgemm_options | None = None):
    lib = load()
    h = _vp()
    if options is None:
        rc = lib.spgemm_create(ctypes.byref(h), m, k, n, ctypes.byref(A), ctypes.byref(B), _vp(stream))
    else:
        rc = lib.spgemm_create_ex(ctypes.byref(h), m, k, n, ctypes.byref(A), ctypes.byref(B), _vp(stream),
                                  ctypes.byref(options))
    _check(rc, "spgemm_create")
    return h


def spgemm_symbolic(h, c_row_ptr: int) -> int:
    nnz = _i64(0)
    _check(load().spgemm_symbolic(h, _vp(c_row_ptr), ctypes.byref(nnz)), "spgemm_symbolic")
    return nnz.value


def spgemm_numeric(h, c_col: int, c_val: int):
    _check(load().spgemm_numeric(h, _vp(c_col), _vp(c_val)), "spgemm_numeric")


def spgemm_numeric_rows(h, row_begin: int, row_end: int, c_col: int, c_val: int):
    _check(load().spgemm_numeric_rows(h, row_begin, row_end, _vp(c_col), _vp(c_val)),
           "spgemm_numeric_rows")


def spgemm_numeric_host(h, c_row_ptr: int, c_col: int, c_val: int, window_nnz: int = 0):
    _check(load().spgemm_numeric_host(h, _vp(c_row_ptr) if c_row_ptr else None, _vp(c_col), _vp(c_val),
                                      window_nnz), "spgemm_numeric_host")


def spgemm_row_windows(h, target_nnz: int = 0):
    """Row cuts of a windowed numeric phase and the entries of C in its largest window."""
    n = _i64(0)
    wmax = _i64(0)
    rc = load().spgemm_row_windows(h, target_nnz, None, 0, ctypes.byref(n), ctypes.byref(wmax))
    if rc != 0 and n.value <= 0:
        _check(rc, "spgemm_row_windows")
    cuts = (_i64 * (n.value + 1))()
    _check(load().spgemm_row_windows(h, target_nnz, cuts, n.value + 1, ctypes.byref(n), ctypes.byref(wmax)),
           "spgemm_row_windows")
    return [int(x) for x in cuts], int(wmax.value)


def spgemm_get_stats(h) -> spgemm_stats:
    s = spgemm_stats()
    _check(load().spgemm_get_stats(h, ctypes.byref(s)), "spgemm_get_stats")
    return s


def spgemm_get_plan(h) -> spgemm_plan:
    p = spgemm_plan()
    _check(load().spgemm_get_plan(h, ctypes.byref(p)), "spgemm_get_plan")
    return p


def spgemm_get_phase_times(h):
    """{phase name: (milliseconds, timed regions)} since create (needs FLAG_TIMING)."""
    n = len(PHASES)
    t = (ctypes.c_double * n)()
    c = (ctypes.c_int64 * n)()
    _check(load().spgemm_get_phase_times(h, t, c, n), "spgemm_get_phase_times")
    return {PHASES[i]: (t[i], c[i]) for i in range(n)}


def spgemm_kernel_launches() -> int:
    return int(load().spgemm_kernel_launches())


def spgemm_symbolic_noalloc(m, k, n, A: spgemm_csr, B: spgemm_csr, c_row_ptr: int, stream: int = 0) -> int:
    """C.row_ptr and nnz(C) without device allocation (light products only; see spgemm.h)."""
    nnz = _i64(0)
    _check(load().spgemm_symbolic_noalloc(m, k, n, ctypes.byref(A), ctypes.byref(B), _vp(c_row_ptr),
                                          ctypes.byref(nnz), _vp(stream)), "spgemm_symbolic_noalloc")
    return nnz.value


def spgemm_hll_estimate(A: spgemm_csr, B: spgemm_csr, registers: int, coef: float, cap: int, stream: int = 0):
    """HyperLogLog capacity of every row of A*B into the device array ``cap`` (see spgemm.h)."""
    _check(load().spgemm_hll_estimate(ctypes.byref(A), ctypes.byref(B), registers, coef, _vp(cap), _vp(stream)),
           "spgemm_hll_estimate")


def spgemm_mcl_prune_symbolic(C: spgemm_csr, threshold: float, col_sums: int, out_row_ptr: int, stream: int = 0) -> int:
    """Column sums and the pruned row offsets of a Markov-clustering step; returns the pruned nnz."""
    nnz = _i64(0)
    _check(load().spgemm_mcl_prune_symbolic(ctypes.byref(C), threshold, _vp(col_sums), _vp(out_row_ptr),
                                            ctypes.byref(nnz), _vp(stream)), "spgemm_mcl_prune_symbolic")
    return nnz.value


def spgemm_mcl_prune_numeric(C: spgemm_csr, threshold: float, col_sums: int, out_row_ptr: int, out_col: int,
                             out_val: int, stream: int = 0):
    _check(load().spgemm_mcl_prune_numeric(ctypes.byref(C), threshold, _vp(col_sums), _vp(out_row_ptr),
                                           _vp(out_col), _vp(out_val), _vp(stream)), "spgemm_mcl_prune_numeric")


def spgemm_destroy(h):
    _check(load().spgemm_destroy(h), "spgemm_destroy")


def spgemm_release_memory():
    _check(load().spgemm_release_memory(), "spgemm_release_memory")


def spgemm_strerror(code: int) -> str:
    return load().spgemm_strerror(code).decode()


def spgemm_last_error() -> str:
    return load().spgemm_last_error().decode()


def options(**kw) -> spgemm_options:
    o = spgemm_options()
    for k, v in kw.items():
        setattr(o, k, v)
    return o
