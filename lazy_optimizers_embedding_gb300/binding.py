"""Thin ctypes binding of libsparseopt (include/sparseopt.h).

Argument marshalling only: every function passes tensor data pointers, sizes and
the current CUDA stream to the C entry point of the same name and returns its
status code.  All work runs in the library's kernels; PyTorch only supplies the
device memory and the stream.  There is no fallback: if the library is not
built, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

OK = 0
ERR_INVALID_ARG = 1
ERR_INDEX_OUT_OF_RANGE = 2
ERR_NOT_CANONICAL = 3
ERR_STEP_ORDER = 4
ERR_WORKSPACE = 5
ERR_CUDA = 6
ERR_INTERNAL = 7
ERR_NON_FINITE = 8
ERR_BAD_STATE = 9

LAZY = 0
DORMANCY_DECAY = 1
WD_L2 = 0          # sparse_adam_wd_mode_t
WD_DECOUPLED = 1
LAST_STEP_PER_ROW = 0
LAST_STEP_PER_COORD = 1
GRAD_ROW_COO = 0
GRAD_CSR = 1


class AdamConfig(ctypes.Structure):
    """sparse_adam_config_t (SparseAdamConfig); weight decay 0 and mode WD_L2 unless given."""
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double), ("weight_decay_mode", ctypes.c_int32)]


class SgdConfig(ctypes.Structure):
    """sparse_sgd_config_t (SparseSgdConfig)."""
    _fields_ = [("lr", ctypes.c_double), ("momentum", ctypes.c_double), ("weight_decay", ctypes.c_double)]


class Grad(ctypes.Structure):
    """sparse_grad_t: a row-COO or CSR gradient (device arrays)."""
    _fields_ = [("form", ctypes.c_int), ("n", ctypes.c_int64), ("row_idx", ctypes.c_void_p),
                ("row_off", ctypes.c_void_p), ("cols", ctypes.c_void_p), ("vals", ctypes.c_void_p),
                ("is_canonical", ctypes.c_int)]


class SparseOptError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        super().__init__(f"{where}: {status_string(code)} (status {code})")
        self.code = code


def _load():
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"libsparseopt.so is not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I64, INT, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    sig = {
        "sparse_workspace_size": (SZ, [I64, I64, I64]),
        "sparse_status_string": (ctypes.c_char_p, [INT]),
        "sparse_canonicalize": (INT, [P, P, I64, I64, I64, P, P, P, P, P, P, SZ, P, P]),
        "sparse_csr_to_coo": (INT, [P, P, I64, I64, I64, P, P, P]),
        "sparse_coo_to_csr": (INT, [P, I64, I64, I64, P, P, P, P]),
        "sparse_row_coo_to_csr": (INT, [P, I64, I64, I64, P, P, P, P]),
        "sparse_adam_step": (INT, [P, P, P, P, I64, P, P, I64, INT, I64, AdamConfig, INT, P, SZ, P, P]),
        "sparse_adam_table_step": (INT, [P, P, P, P, INT, I64, I64, ctypes.POINTER(Grad), I64, AdamConfig,
                                         INT, P, SZ, P, P]),
        "sparse_sgd_step": (INT, [P, P, I64, P, P, I64, INT, SgdConfig, P, SZ, P, P]),
        "sparse_sgd_table_step": (INT, [P, P, I64, I64, ctypes.POINTER(Grad), SgdConfig, P, SZ, P, P]),
        "sparse_canonicalize_static_ws": (INT, [P, P, I64, I64, I64, P, P, P, P, P, P, P]),
        "sparse_read_rows": (INT, [P, I64, I64, P, I64, P, P, P]),
        "sparse_check_finite": (INT, [P, I64, P, P]),
        "sparse_check_state": (INT, [P, P, I64, I64, ctypes.POINTER(Grad), P, P]),
        "sparse_profile_enable": (None, [INT]),
        "sparse_profile_reset": (None, []),
        "sparse_profile_read": (INT, [INT, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_int64),
                                      ctypes.POINTER(ctypes.c_double)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


LIB = _load()
EXPORTED = ("sparse_workspace_size", "sparse_status_string", "sparse_canonicalize", "sparse_csr_to_coo",
            "sparse_coo_to_csr", "sparse_row_coo_to_csr", "sparse_adam_step", "sparse_adam_table_step",
            "sparse_sgd_step", "sparse_sgd_table_step", "sparse_canonicalize_static_ws", "sparse_profile_enable",
            "sparse_profile_reset", "sparse_profile_read", "sparse_read_rows", "sparse_check_finite",
            "sparse_check_state")
STATIC_WS_BYTES = 16 * 1024 * 1024  # SPARSE_STATIC_WS_BYTES


# ------------------------------------------------------------------ marshalling
def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ws(ws):
    if ws is None:
        return None, 0
    return _ptr(ws, torch.uint8, "ws"), ws.numel()


def status_string(code: int) -> str:
    return LIB.sparse_status_string(int(code)).decode()


sparse_status_string = status_string


def check(code: int, where: str = "") -> None:
    if code != OK:
        raise SparseOptError(code, where)


def sparse_workspace_size(n: int, c: int, bound: int) -> int:
    return int(LIB.sparse_workspace_size(int(n), int(c), int(bound)))


def workspace(n: int, c: int, bound: int, device="cuda") -> torch.Tensor:
    """Device workspace for raw inputs of up to n entries of width c, keys < bound."""
    return torch.empty(max(sparse_workspace_size(n, c, bound), 256), dtype=torch.uint8, device=device)


def error_word(device="cuda") -> torch.Tensor:
    """The sticky device error word (int32, zero = no error)."""
    return torch.zeros(1, dtype=torch.int32, device=device)


def row_coo(rows, vals, canonical: bool) -> Grad:
    g = Grad()
    g.form = GRAD_ROW_COO
    g.n = rows.numel()
    g.row_idx = _ptr(rows, torch.int64, "rows")
    g.vals = _ptr(vals, torch.float32, "vals")
    g.is_canonical = int(bool(canonical))
    g._tensors = (rows, vals)  # keep the arrays alive while the struct is in use
    return g


def csr(row_off, cols, vals) -> Grad:
    g = Grad()
    g.form = GRAD_CSR
    g.n = cols.numel()
    g.row_off = _ptr(row_off, torch.int64, "row_off")
    g.cols = _ptr(cols, torch.int32, "cols")
    g.vals = _ptr(vals, torch.float32, "vals")
    g.is_canonical = 1
    g._tensors = (row_off, cols, vals)
    return g


# ------------------------------------------------------------------ entry points
def sparse_canonicalize(idx, vals, n, c, bound, idx_out, vals_out, seg_off_out, perm_out, nnz_out, ws, d_err,
                        stream=None) -> int:
    wp, wb = _ws(ws)
    return LIB.sparse_canonicalize(_ptr(idx, torch.int64, "idx"), _ptr(vals, torch.float32, "vals"), int(n),
                                   int(c), int(bound), _ptr(idx_out, torch.int64, "idx_out"),
                                   _ptr(vals_out, torch.float32, "vals_out"),
                                   _ptr(seg_off_out, torch.int64, "seg_off_out"),
                                   _ptr(perm_out, torch.int64, "perm_out"), _ptr(nnz_out, torch.int64, "nnz_out"),
                                   wp, wb, _ptr(d_err, torch.int32, "d_err"), _stream(stream))


def sparse_canonicalize_static_ws(idx, vals, n, c, bound, idx_out, vals_out, seg_off_out, perm_out, nnz_out, d_err,
                                  stream=None) -> int:
    """sparse_canonicalize with the library's fixed device scratch array instead of a workspace:
    for callers that cannot allocate device memory (see include/sparseopt.h for the size limit and
    the rule that calls must not overlap on the GPU)."""
    return LIB.sparse_canonicalize_static_ws(_ptr(idx, torch.int64, "idx"), _ptr(vals, torch.float32, "vals"),
                                             int(n), int(c), int(bound), _ptr(idx_out, torch.int64, "idx_out"),
                                             _ptr(vals_out, torch.float32, "vals_out"),
                                             _ptr(seg_off_out, torch.int64, "seg_off_out"),
                                             _ptr(perm_out, torch.int64, "perm_out"),
                                             _ptr(nnz_out, torch.int64, "nnz_out"), _ptr(d_err, torch.int32, "d_err"),
                                             _stream(stream))


def sparse_csr_to_coo(row_off, cols, r, c, nnz, lin_out, d_err, stream=None) -> int:
    return LIB.sparse_csr_to_coo(_ptr(row_off, torch.int64, "row_off"), _ptr(cols, torch.int32, "cols"), int(r),
                                 int(c), int(nnz), _ptr(lin_out, torch.int64, "lin_out"),
                                 _ptr(d_err, torch.int32, "d_err"), _stream(stream))


def sparse_coo_to_csr(lin, nnz, r, c, row_off_out, cols_out, d_err, stream=None) -> int:
    return LIB.sparse_coo_to_csr(_ptr(lin, torch.int64, "lin"), int(nnz), int(r), int(c),
                                 _ptr(row_off_out, torch.int64, "row_off_out"),
                                 _ptr(cols_out, torch.int32, "cols_out"), _ptr(d_err, torch.int32, "d_err"),
                                 _stream(stream))


def sparse_row_coo_to_csr(rows, nrows, r, c, row_off_out, cols_out, d_err, stream=None) -> int:
    return LIB.sparse_row_coo_to_csr(_ptr(rows, torch.int64, "rows"), int(nrows), int(r), int(c),
                                     _ptr(row_off_out, torch.int64, "row_off_out"),
                                     _ptr(cols_out, torch.int32, "cols_out"), _ptr(d_err, torch.int32, "d_err"),
                                     _stream(stream))


def sparse_adam_step(p, m, v, last_step, dim, idx, g, nnz, is_canonical, t, cfg: AdamConfig, mode, ws, d_err,
                     stream=None) -> int:
    wp, wb = _ws(ws)
    return LIB.sparse_adam_step(_ptr(p, torch.float32, "p"), _ptr(m, torch.float32, "m"),
                                _ptr(v, torch.float32, "v"), _ptr(last_step, torch.int64, "last_step"), int(dim),
                                _ptr(idx, torch.int64, "idx"), _ptr(g, torch.float32, "g"), int(nnz),
                                int(is_canonical), int(t), cfg, int(mode), wp, wb,
                                _ptr(d_err, torch.int32, "d_err"), _stream(stream))


def sparse_adam_table_step(p, m, v, last_step, ls_layout, r, c, grad: Grad, t, cfg: AdamConfig, mode, ws, d_err,
                           stream=None) -> int:
    wp, wb = _ws(ws)
    return LIB.sparse_adam_table_step(_ptr(p, torch.float32, "p"), _ptr(m, torch.float32, "m"),
                                      _ptr(v, torch.float32, "v"), _ptr(last_step, torch.int64, "last_step"),
                                      int(ls_layout), int(r), int(c), ctypes.byref(grad), int(t), cfg, int(mode),
                                      wp, wb, _ptr(d_err, torch.int32, "d_err"), _stream(stream))


def sparse_sgd_step(p, buf, dim, idx, g, nnz, is_canonical, cfg: SgdConfig, ws, d_err, stream=None) -> int:
    wp, wb = _ws(ws)
    return LIB.sparse_sgd_step(_ptr(p, torch.float32, "p"), _ptr(buf, torch.float32, "buf"), int(dim),
                               _ptr(idx, torch.int64, "idx"), _ptr(g, torch.float32, "g"), int(nnz),
                               int(is_canonical), cfg, wp, wb, _ptr(d_err, torch.int32, "d_err"), _stream(stream))


def sparse_sgd_table_step(p, buf, r, c, grad: Grad, cfg: SgdConfig, ws, d_err, stream=None) -> int:
    wp, wb = _ws(ws)
    return LIB.sparse_sgd_table_step(_ptr(p, torch.float32, "p"), _ptr(buf, torch.float32, "buf"), int(r),
                                     int(c), ctypes.byref(grad), cfg, wp, wb, _ptr(d_err, torch.int32, "d_err"),
                                     _stream(stream))


def sparse_check_finite(vals, n, d_err, stream=None) -> int:
    return LIB.sparse_check_finite(_ptr(vals, torch.float32, "vals"), int(n), _ptr(d_err, torch.int32, "d_err"),
                                   _stream(stream))


def sparse_check_state(m, v, r, c, grad: Grad, d_err, stream=None) -> int:
    return LIB.sparse_check_state(_ptr(m, torch.float32, "m"), _ptr(v, torch.float32, "v"), int(r), int(c),
                                  ctypes.byref(grad), _ptr(d_err, torch.int32, "d_err"), _stream(stream))


def sparse_read_rows(table, r, c, idx, n, out, d_err, stream=None) -> int:
    return LIB.sparse_read_rows(_ptr(table, torch.float32, "table"), int(r), int(c), _ptr(idx, torch.int64, "idx"),
                                int(n), _ptr(out, torch.float32, "out"), _ptr(d_err, torch.int32, "d_err"),
                                _stream(stream))


# ------------------------------------------------------------------ diagnostics
def sparse_profile_enable(enable: bool = True) -> None:
    LIB.sparse_profile_enable(int(bool(enable)))


def sparse_profile_reset() -> None:
    LIB.sparse_profile_reset()


def sparse_profile_read(max_entries: int = 64) -> dict:
    """{kernel name: (launches, total GPU ms)} since the last reset (waits for the recorded events)."""
    names = (ctypes.c_char_p * max_entries)()
    launches = (ctypes.c_int64 * max_entries)()
    ms = (ctypes.c_double * max_entries)()
    n = LIB.sparse_profile_read(max_entries, names, launches, ms)
    return {names[i].decode(): (int(launches[i]), float(ms[i])) for i in range(min(n, max_entries))}
