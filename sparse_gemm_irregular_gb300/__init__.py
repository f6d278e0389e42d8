"""Single-GPU SpGEMM C = A * B on CSR matrices for NVIDIA GB300 (sm_103a).

The product runs in the hand-written CUDA kernels of libspgemm_gb300.so (C ABI in
include/spgemm.h).  This package only marshals arguments: ``DeviceCSR`` keeps a CSR matrix in
PyTorch device tensors, and ``multiply`` drives create / symbolic / numeric / destroy.
"""
from __future__ import annotations

from dataclasses import dataclass

from . import binding
from .binding import (SpgemmError, load, options, spgemm_create, spgemm_destroy, spgemm_get_phase_times,
                      spgemm_hll_estimate, spgemm_mcl_prune_numeric, spgemm_mcl_prune_symbolic,
                      spgemm_numeric_host,
                      spgemm_get_plan, spgemm_get_stats, spgemm_kernel_launches, spgemm_last_error, spgemm_numeric,
                      spgemm_numeric_rows, spgemm_plan_params, spgemm_release_memory, spgemm_row_windows,
                      spgemm_strerror, spgemm_symbolic)

__all__ = [
    "DeviceCSR", "multiply", "Product", "SpgemmError", "load", "options", "spgemm_create",
    "spgemm_destroy", "spgemm_get_phase_times", "spgemm_get_plan", "spgemm_get_stats", "spgemm_hll_estimate",
    "spgemm_mcl_prune_symbolic", "spgemm_mcl_prune_numeric", "mcl_iteration",
    "spgemm_kernel_launches",
    "spgemm_last_error", "spgemm_numeric", "spgemm_numeric_rows", "spgemm_plan_params",
    "spgemm_release_memory", "spgemm_row_windows",
    "spgemm_strerror", "spgemm_symbolic",
]


@dataclass
class DeviceCSR:
    """CSR matrix in device memory: row_ptr int64 (rows+1), col int32 (nnz), val float64 (nnz)."""
    rows: int
    cols: int
    row_ptr: "object"
    col: "object"
    val: "object"

    @property
    def nnz(self) -> int:
        return int(self.col.numel())

    @staticmethod
    def from_host(m, device="cuda", pin: bool = False) -> "DeviceCSR":
        """Upload a host CSR (anything with rows, cols, row_ptr, col, val numpy arrays)."""
        import torch
        def up(a, dt):
            t = torch.from_numpy(a).to(dt)
            if pin:
                t = t.pin_memory()
            return t.to(device, non_blocking=pin)
        return DeviceCSR(m.rows, m.cols, up(m.row_ptr, torch.int64), up(m.col, torch.int32),
                         up(m.val, torch.float64))

    def desc(self) -> binding.spgemm_csr:
        d = binding.spgemm_csr()
        d.rows, d.cols, d.nnz = self.rows, self.cols, self.nnz
        d.row_ptr = self.row_ptr.data_ptr()
        d.col_idx = self.col.data_ptr() if self.nnz else 0
        d.vals = self.val.data_ptr() if self.nnz else 0
        return d

    def to_host(self):
        """(row_ptr, col, val) as numpy arrays."""
        return self.row_ptr.cpu().numpy(), self.col.cpu().numpy(), self.val.cpu().numpy()


class Product:
    """One product C = A * B: the handle plus the caller-owned C arrays."""

    def __init__(self, A: DeviceCSR, B: DeviceCSR, stream=None, opts=None):
        import torch
        self.A, self.B = A, B
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        self._da, self._db = A.desc(), B.desc()  # kept alive: the library borrows the pointers
        self.h = spgemm_create(A.rows, A.cols, B.cols, self._da, self._db, self.stream.cuda_stream, opts)
        self.row_ptr = None
        self.nnz = None

    def symbolic(self):
        import torch
        self.row_ptr = torch.empty(self.A.rows + 1, dtype=torch.int64, device=self.A.row_ptr.device)
        self.nnz = spgemm_symbolic(self.h, self.row_ptr.data_ptr())
        return self.row_ptr, self.nnz

    def numeric(self, col=None, val=None):
        import torch
        dev = self.A.row_ptr.device
        if col is None:
            col = torch.empty(max(self.nnz, 1), dtype=torch.int32, device=dev)
        if val is None:
            val = torch.empty(max(self.nnz, 1), dtype=torch.float64, device=dev)
        spgemm_numeric(self.h, col.data_ptr(), val.data_ptr())
        return col[:self.nnz], val[:self.nnz]

    def numeric_rows(self, row_begin: int, row_end: int, col, val):
        spgemm_numeric_rows(self.h, row_begin, row_end, col.data_ptr(), val.data_ptr())

    def row_windows(self, target_nnz: int = 0):
        """(row cuts, entries of C in the largest window) for numeric_rows window by window."""
        return spgemm_row_windows(self.h, target_nnz)

    def numeric_windows(self, col, val, target_nnz: int = 0, cuts=None):
        """Numeric phase window by window into the same device arrays col / val (each window at
        offset 0; they need the largest window's entries).  Returns the cuts used."""
        if cuts is None:
            cuts, wmax = self.row_windows(target_nnz)
            if col.numel() < wmax or val.numel() < wmax:
                raise ValueError("window buffers shorter than the largest window")
        for rb, re in zip(cuts[:-1], cuts[1:]):
            spgemm_numeric_rows(self.h, rb, re, col.data_ptr(), val.data_ptr())
        return cuts

    def numeric_host(self, col, val, row_ptr=None, window_nnz: int = 0):
        """Numeric phase into host (CPU) tensors col (int32, nnz) and val (float64, nnz), and
        row_ptr (int64, rows+1) when given; pinned tensors reach the full copy bandwidth."""
        for t in (col, val) + ((row_ptr,) if row_ptr is not None else ()):
            if t.device.type != "cpu" or not t.is_contiguous():
                raise ValueError("numeric_host wants contiguous CPU tensors")
        if col.numel() < self.nnz or val.numel() < self.nnz:
            raise ValueError("host arrays shorter than nnz(C)")
        spgemm_numeric_host(self.h, row_ptr.data_ptr() if row_ptr is not None else 0, col.data_ptr(),
                            val.data_ptr(), window_nnz)

    def stats(self):
        return spgemm_get_stats(self.h)

    def plan(self):
        return spgemm_get_plan(self.h)

    def phase_times(self):
        return spgemm_get_phase_times(self.h)

    def close(self):
        if self.h is not None:
            spgemm_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def multiply(A: DeviceCSR, B: DeviceCSR, stream=None, opts=None) -> DeviceCSR:
    """C = A * B, all on the device; returns C as a DeviceCSR."""
    p = Product(A, B, stream, opts)
    try:
        row_ptr, _ = p.symbolic()
        col, val = p.numeric()
    finally:
        p.close()
    return DeviceCSR(A.rows, B.cols, row_ptr, col, val)


def mcl_iteration(M: DeviceCSR, threshold: float = 0.002, stream=None, opts=None) -> DeviceCSR:
    """One Markov-clustering iteration (Trident page, section 5.7): the expansion M * M on the
    library's SpGEMM, then column normalization, pruning below ``threshold`` and the element-wise
    square, all on the device.  Returns the new matrix."""
    import torch
    p = Product(M, M, stream=stream, opts=opts)
    try:
        p.symbolic()
        col, val = p.numeric()
        C = DeviceCSR(M.rows, M.cols, p.row_ptr, col, val)
    finally:
        p.close()
    dev = M.row_ptr.device
    st = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
    sums = torch.empty(max(M.cols, 1), dtype=torch.float64, device=dev)
    rp = torch.empty(M.rows + 1, dtype=torch.int64, device=dev)
    cd = C.desc()
    nnz = spgemm_mcl_prune_symbolic(cd, threshold, sums.data_ptr(), rp.data_ptr(), st)
    oc = torch.empty(max(nnz, 1), dtype=torch.int32, device=dev)
    ov = torch.empty(max(nnz, 1), dtype=torch.float64, device=dev)
    spgemm_mcl_prune_numeric(cd, threshold, sums.data_ptr(), rp.data_ptr(), oc.data_ptr(), ov.data_ptr(), st)
    return DeviceCSR(M.rows, M.cols, rp, oc[:nnz], ov[:nnz])
