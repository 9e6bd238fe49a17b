"""CPU oracle for the sparse / lazy optimizer step -- TEST INFRASTRUCTURE.

Plain, slow, obviously correct: the C functions in ``sparse_oracle.c`` (fp64
arithmetic, scalar loops, a library sort) plus the tiny dense emulator in
``dense_emulator.py``.  Only the tests, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU baseline / reference arm may import this package; the product
(``lazy_optimizers_embedding_gb300``) never does, and the two share no code.

Status codes: 0 ok, 1 invalid argument, 2 index out of range, 3 not canonical,
4 step order (t <= last_step), 8 non-finite gradient value, 9 corrupted moment
state (NaN / infinite m or v, negative v), 100 out of host memory.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sparse_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libsparse_oracle.so")

MODE_LAZY = 0
MODE_DORMANCY_DECAY = 1
WD_L2 = 0          # weight decay added to the gradient (classic Adam L2)
WD_DECOUPLED = 1   # weight decay added to the descent direction (AdamW)
LS_PER_ROW = 0
LS_PER_COORD = 1
FORM_ROW_COO = 0
FORM_CSR = 1

OK, ERR_INVALID_ARG, ERR_INDEX_OUT_OF_RANGE, ERR_NOT_CANONICAL, ERR_STEP_ORDER = 0, 1, 2, 3, 4
ERR_NON_FINITE = 8
ERR_BAD_STATE = 9


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction: the same on x86 and Arm)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_D = ctypes.c_double


def lib():
    global _lib
    if _lib is None:
        l = ctypes.CDLL(build())
        l.oracle_canonicalize.argtypes = [_P, _P, _I64, _I64, _I64, _P, _P, _P, _P, _P]
        l.oracle_csr_validate.argtypes = [_P, _P, _I64, _I64, _I64, _INT]
        l.oracle_csr_to_coo.argtypes = [_P, _P, _I64, _I64, _I64, _P]
        l.oracle_coo_to_csr.argtypes = [_P, _I64, _I64, _I64, _P, _P]
        l.oracle_row_coo_to_csr.argtypes = [_P, _I64, _I64, _I64, _P, _P]
        l.oracle_adam_table_step.argtypes = [_P, _P, _P, _INT, _P, _INT, _I64, _I64, _INT,
                                             _P, _I64, _INT, _P, _P, _P,
                                             _I64, _D, _D, _D, _D, _INT, _D, _INT]
        l.oracle_read_rows.argtypes = [_P, _I64, _I64, _P, _I64, _P]
        l.oracle_check_finite.argtypes = [_P, _I64]
        l.oracle_check_finite.restype = _INT
        l.oracle_check_state.argtypes = [_P, _P, _I64, _I64, _INT, _P, _I64, _P, _P]
        l.oracle_check_state.restype = _INT
        l.oracle_read_rows.restype = _INT
        l.oracle_sgd_table_step.argtypes = [_P, _P, _INT, _I64, _I64, _INT,
                                            _P, _I64, _INT, _P, _P, _P, _D, _D, _D]
        for f in (l.oracle_canonicalize, l.oracle_csr_validate, l.oracle_csr_to_coo,
                  l.oracle_coo_to_csr, l.oracle_row_coo_to_csr, l.oracle_adam_table_step,
                  l.oracle_sgd_table_step):
            f.restype = ctypes.c_int
        _lib = l
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: oracle status {code}")
        self.code = code


def canonicalize(idx, vals, bound: int, *, check=True):
    """Raw COO -> canonical COO.  Returns (idx_out, vals_out, seg_off, perm) or the status code."""
    idx = _c(idx, np.int64)
    vals = _c(vals, np.float32)
    n = idx.shape[0]
    c = 1 if vals.ndim == 1 else vals.shape[1]
    idx_out = np.empty(max(n, 1), np.int64)
    vals_out = np.empty((max(n, 1), c), np.float32)
    seg = np.empty(n + 1, np.int64)
    perm = np.empty(max(n, 1), np.int64)
    nnz = np.zeros(1, np.int64)
    rc = lib().oracle_canonicalize(_ptr(idx), _ptr(vals), n, c, bound, _ptr(idx_out),
                                   _ptr(vals_out), _ptr(seg), _ptr(perm), _ptr(nnz))
    if rc:
        if check:
            raise OracleError(rc, "canonicalize")
        return rc
    u = int(nnz[0])
    vo = vals_out[:u] if vals.ndim > 1 else vals_out[:u, 0]
    return idx_out[:u].copy(), vo.copy(), seg[:u + 1].copy(), perm[:n].copy()


def csr_to_coo(row_off, cols, r: int, c: int, *, check=True):
    row_off = _c(row_off, np.int64)
    cols = _c(cols, np.int32)
    nnz = cols.shape[0]
    lin = np.empty(max(nnz, 1), np.int64)
    rc = lib().oracle_csr_to_coo(_ptr(row_off), _ptr(cols), r, c, nnz, _ptr(lin))
    if rc:
        if check:
            raise OracleError(rc, "csr_to_coo")
        return rc
    return lin[:nnz].copy()


def coo_to_csr(lin, r: int, c: int, *, check=True):
    lin = _c(lin, np.int64)
    nnz = lin.shape[0]
    row_off = np.empty(r + 1, np.int64)
    cols = np.empty(max(nnz, 1), np.int32)
    rc = lib().oracle_coo_to_csr(_ptr(lin), nnz, r, c, _ptr(row_off), _ptr(cols))
    if rc:
        if check:
            raise OracleError(rc, "coo_to_csr")
        return rc
    return row_off, cols[:nnz].copy()


def row_coo_to_csr(rows, r: int, c: int, *, check=True):
    rows = _c(rows, np.int64)
    nr = rows.shape[0]
    row_off = np.empty(r + 1, np.int64)
    cols = np.empty(max(nr * c, 1), np.int32)
    rc = lib().oracle_row_coo_to_csr(_ptr(rows), nr, r, c, _ptr(row_off), _ptr(cols))
    if rc:
        if check:
            raise OracleError(rc, "row_coo_to_csr")
        return rc
    return row_off, cols[:nr * c].copy()


def _state_kind(*arrs):
    dt = arrs[0].dtype
    for a in arrs:
        if a is None:
            continue
        assert a.dtype == dt and a.flags.c_contiguous, "state arrays must share a dtype and be contiguous"
    assert dt in (np.float32, np.float64)
    return int(dt == np.float64)


def adam_table_step(p, m, v, last_step, t: int, *, lr, beta1, beta2, eps, mode,
                    rows=None, vals=None, is_canonical=False, row_off=None, cols=None,
                    ls_per_coord=False, weight_decay=0.0, wd_mode=0) -> int:
    """One lazy Adam step, in place on p, m, v ([r, c] or [r]) and last_step.  Returns the status.

    Gradient as row-COO (``rows``, ``vals`` [n, c]) or CSR (``row_off``, ``cols``, ``vals`` [nnz]).
    """
    f64 = _state_kind(p, m, v)
    r = p.shape[0]
    c = 1 if p.ndim == 1 else p.shape[1]
    assert last_step.dtype == np.int64 and last_step.flags.c_contiguous
    if row_off is not None:
        form, n = FORM_CSR, _c(cols, np.int32).shape[0]
        row_off, cols, vals = _c(row_off, np.int64), _c(cols, np.int32), _c(vals, np.float32)
        rows = None
    else:
        form = FORM_ROW_COO
        rows, vals = _c(rows, np.int64), _c(vals, np.float32)
        n = rows.shape[0]
    return lib().oracle_adam_table_step(
        _ptr(p), _ptr(m), _ptr(v), f64, _ptr(last_step), LS_PER_COORD if ls_per_coord else LS_PER_ROW,
        r, c, form, _ptr(rows), n, int(bool(is_canonical)), _ptr(row_off), _ptr(cols), _ptr(vals),
        int(t), float(lr), float(beta1), float(beta2), float(eps), int(mode), float(weight_decay), int(wd_mode))


def check_finite(vals) -> int:
    """ERR_NON_FINITE when any value is NaN or infinite, else OK."""
    vals = _c(vals, np.float32)
    return lib().oracle_check_finite(_ptr(vals), vals.size)


def check_state(m, v, *, rows=None, row_off=None, cols=None) -> int:
    """Validation of the Adam moments a step would read ("DiskSparseAdam (DSA)" README,
    "Validated Inputs": NaN / negative moment rows).  m, v: [r, c] (or [dim]) fp32;
    the gradient's structure as row-COO rows (any order, repeats allowed) or CSR
    (row_off, cols).  Returns ERR_BAD_STATE, ERR_INDEX_OUT_OF_RANGE, ERR_NOT_CANONICAL
    (malformed CSR) or OK."""
    m, v = _c(m, np.float32), _c(v, np.float32)
    assert m.shape == v.shape
    r = m.shape[0]
    c = 1 if m.ndim == 1 else m.shape[1]
    if row_off is not None:
        row_off, cols = _c(row_off, np.int64), _c(cols, np.int32)
        return lib().oracle_check_state(_ptr(m), _ptr(v), r, c, FORM_CSR, None, cols.shape[0], _ptr(row_off),
                                        _ptr(cols))
    rows = _c(rows, np.int64)
    return lib().oracle_check_state(_ptr(m), _ptr(v), r, c, FORM_ROW_COO, _ptr(rows), rows.shape[0], None, None)


def read_rows(table, idx, *, check=True):
    """The rows of a [r, c] fp32 table at the given indices, bit for bit ([n, c])."""
    table = _c(table, np.float32)
    r = table.shape[0]
    c = 1 if table.ndim == 1 else table.shape[1]
    idx = _c(idx, np.int64)
    out = np.empty((idx.shape[0], c), np.float32)
    rc = lib().oracle_read_rows(_ptr(table), r, c, _ptr(idx), idx.shape[0], _ptr(out))
    if rc:
        if check:
            raise OracleError(rc, "read_rows")
        return rc
    return out


def sgd_table_step(p, buf, *, lr, momentum, weight_decay, rows=None, vals=None,
                   is_canonical=False, row_off=None, cols=None) -> int:
    """One sparse SGD step, in place on p (and buf when momentum > 0).  Returns the status."""
    f64 = _state_kind(p, buf)
    r = p.shape[0]
    c = 1 if p.ndim == 1 else p.shape[1]
    if row_off is not None:
        form, n = FORM_CSR, _c(cols, np.int32).shape[0]
        row_off, cols, vals = _c(row_off, np.int64), _c(cols, np.int32), _c(vals, np.float32)
        rows = None
    else:
        form = FORM_ROW_COO
        rows, vals = _c(rows, np.int64), _c(vals, np.float32)
        n = rows.shape[0]
    return lib().oracle_sgd_table_step(
        _ptr(p), _ptr(buf), f64, r, c, form, _ptr(rows), n, int(bool(is_canonical)),
        _ptr(row_off), _ptr(cols), _ptr(vals), float(lr), float(momentum), float(weight_decay))


def adam_step(p, m, v, last_step, idx, g, t: int, *, is_canonical=True, **cfg) -> int:
    """1-D lazy Adam: the table step with one column (last_step per coordinate)."""
    return adam_table_step(p, m, v, last_step, t, rows=idx, vals=np.asarray(g).reshape(-1, 1),
                           is_canonical=is_canonical, **cfg)


def sgd_step(p, buf, idx, g, *, is_canonical=True, **cfg) -> int:
    """1-D sparse SGD: the table step with one column."""
    return sgd_table_step(p, buf, rows=idx, vals=np.asarray(g).reshape(-1, 1),
                          is_canonical=is_canonical, **cfg)
