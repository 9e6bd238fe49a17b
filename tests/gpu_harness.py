"""Shared helpers of the GPU parity tests: run a step sequence through the C-ABI
(binding) and the same sequence through the CPU oracle, then compare.

Tolerances (fp32 state against the fp64 oracle rounded to fp32):
  - p, m, v, buf: |gpu - ref| <= max(1e-5 |ref|, 1e-7) on every coordinate;
  - v also with NO absolute floor: |gpu - ref| <= 1e-5 |ref| on every touched
    coordinate (every term of the second-moment recursion is >= 0, so nothing
    cancels and a relative bound holds at any scale; with gradients of 0.01 the
    floor alone would accept any v in [0, 2e-7]);
  - m also against the scale its rounding errors live on: |gpu - ref| <= 1e-5 M,
    where M is the same recursion run on magnitudes (M = b1 M + (1-beta1)|g|,
    |g| + wd|p| under L2 weight decay).  m's two terms can cancel, so its
    error is bounded relative to M, not to |m|; where M <= 10 |m| (at most one
    decimal digit lost to cancellation) the plain no-floor relative error is
    asserted too;
  - untouched coordinates (planted NaN payloads, -0.0, denormals, infinities
    included) and last_step bit for bit;
  - every device array sits inside a guard region of seeded canary bytes that
    must be unchanged after every call.
The largest errors seen are collected in DIAG and printed in pytest's terminal
summary.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

RTOL = 1e-5
ATOL = 1e-7
MOMENT_RTOL = 1e-5     # v relative (no floor) and m relative to its magnitude scale M
CANCEL = 10.0          # entries with M <= CANCEL*|m| also get the no-floor relative check on m

DIAG: dict[str, dict[str, float]] = {}


def note(key: str, quantity: str, value: float) -> None:
    d = DIAG.setdefault(key, {})
    d[quantity] = max(d.get(quantity, 0.0), float(value))


def tol_violations(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    g = got.astype(np.float64)
    r = ref.astype(np.float64)
    bad = ~(np.abs(g - r) <= np.maximum(RTOL * np.abs(r), ATOL))
    both_nan = np.isnan(g) & np.isnan(r)
    return bad & ~both_nan


def assert_state_close(name, got, ref, touched_mask=None, init=None):
    got = np.asarray(got)
    ref = np.asarray(ref)
    if touched_mask is not None and init is not None:
        un = ~touched_mask
        assert got[un].tobytes() == np.asarray(init)[un].tobytes(), f"{name}: untouched coordinates changed"
        got, ref = got[touched_mask], ref[touched_mask]
    bad = tol_violations(got, ref)
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} outside tolerance; first {i.tolist()}: "
                             f"gpu {got[tuple(i.T)]} ref {ref[tuple(i.T)]}")


def max_rel(got, ref):
    g = np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    nz = r != 0
    return float(np.max(np.abs(g[nz] - r[nz]) / np.abs(r[nz]))) if nz.any() else 0.0


def assert_v_relative(key, name, got, ref, touched):
    """Second moments: no-floor relative error on touched coordinates; exact zeros stay zero."""
    g = np.asarray(got)[touched].astype(np.float64)
    r = np.asarray(ref)[touched].astype(np.float64)
    nz = r != 0
    rel = float(np.max(np.abs(g[nz] - r[nz]) / r[nz])) if nz.any() else 0.0
    note(key, "v max rel (no floor)", rel)
    assert rel <= MOMENT_RTOL, f"{name}: max relative error of v {rel:.3e} > {MOMENT_RTOL}"
    assert np.all(g[~nz] == 0.0), f"{name}: v not zero where the oracle's is"
    return rel


def assert_m_scaled(key, name, got, ref, scale, touched):
    """First moments: error relative to the magnitude scale M, and no-floor relative where
    the recursion did not cancel heavily."""
    g = np.asarray(got)[touched].astype(np.float64)
    r = np.asarray(ref)[touched].astype(np.float64)
    M = np.asarray(scale, np.float64)[touched]
    pos = M > 0
    err = np.abs(g - r)
    worst = float(np.max(err[pos] / M[pos])) if pos.any() else 0.0
    note(key, "m max err / M", worst)
    assert worst <= MOMENT_RTOL, f"{name}: m error {worst:.3e} of its magnitude scale > {MOMENT_RTOL}"
    assert np.all(g[~pos] == r[~pos]), f"{name}: m differs where every gradient was zero"
    well = pos & (np.abs(r) > 0) & (M <= CANCEL * np.abs(r))
    rel = float(np.max(err[well] / np.abs(r[well]))) if well.any() else 0.0
    note(key, "m max rel (no floor, M <= 10|m|)", rel)
    assert rel <= MOMENT_RTOL, f"{name}: max relative error of m {rel:.3e} > {MOMENT_RTOL}"


class MomentScale:
    """M, the scale of m's rounding errors: the oracle's first-moment recursion (fp64 state)
    fed the magnitudes of each step's canonical gradient, |g| (+ wd |p| under L2 decay)."""

    def __init__(self, shape, ls_n, hp, mode, ls_per_coord):
        self.M = np.zeros(shape, np.float64)
        self._p = np.zeros(shape, np.float64)
        self._v = np.zeros(shape, np.float64)
        self._ls = np.zeros(ls_n, np.int64)
        self.hp = dict(hp)
        self.l2 = self.hp.get("weight_decay", 0.0) > 0 and self.hp.get("wd_mode", oracle.WD_L2) == oracle.WD_L2
        self.mode = mode
        self.per_coord = ls_per_coord

    def step(self, t, p_before, *, rows=None, vals=None, is_canonical=True, row_off=None, cols=None):
        self._p[...] = np.abs(p_before) if self.l2 else 0.0
        kw = dict(self.hp, mode=self.mode, ls_per_coord=self.per_coord)
        if row_off is not None:
            rc = oracle.adam_table_step(self._p, self.M, self._v, self._ls, t, row_off=row_off, cols=cols,
                                        vals=np.abs(vals), **kw)
        else:
            if not is_canonical:
                rows, vals = oracle.canonicalize(rows, vals, self.M.shape[0])[:2]
            rc = oracle.adam_table_step(self._p, self.M, self._v, self._ls, t, rows=rows,
                                        vals=np.abs(vals).reshape(rows.shape[0], -1), is_canonical=True, **kw)
        assert rc == 0


# ---------------------------------------------------------------- guard regions
GUARD = 4096   # canary bytes before and after every guarded array (keeps 256-byte alignment)


class Guarded:
    """Device arrays carved out of larger buffers whose padding before and after holds seeded
    random bytes; check() verifies every padding byte after a call, so a write past either
    end of an array (state, gradient, outputs, workspace, error word) is caught."""

    def __init__(self, seed=0, device="cuda"):
        self.items = []
        self.rng = np.random.default_rng(seed)
        self.device = device

    def empty(self, shape, dtype):
        shape = tuple(int(s) for s in (shape if isinstance(shape, (tuple, list)) else (shape,)))
        item = torch.empty((), dtype=dtype).element_size()
        nbytes = int(np.prod(shape, dtype=np.int64)) * item
        body = (nbytes + 255) // 256 * 256
        total = GUARD + body + GUARD
        buf = torch.empty(total, dtype=torch.uint8, device=self.device)
        head = self.rng.integers(0, 256, GUARD, dtype=np.uint8)
        tail = self.rng.integers(0, 256, total - GUARD - nbytes, dtype=np.uint8)
        buf[:GUARD].copy_(torch.from_numpy(head))
        buf[GUARD + nbytes:].copy_(torch.from_numpy(tail))
        self.items.append((buf, nbytes, head, tail))
        if nbytes == 0:
            return buf[GUARD:GUARD].view(dtype).reshape(shape)
        return buf[GUARD:GUARD + nbytes].view(dtype).view(shape)

    def array(self, a, dtype=None):
        a = np.ascontiguousarray(a if dtype is None else np.asarray(a, dtype))
        t = self.empty(a.shape, getattr(torch, a.dtype.name))
        if a.size:
            t.copy_(torch.from_numpy(a))
        return t

    def zeros(self, shape, dtype=torch.float32):
        t = self.empty(shape, dtype)
        t.zero_()
        return t

    def workspace(self, so, n, c, bound):
        return self.empty(max(int(so.sparse_workspace_size(n, c, bound)), 1), torch.uint8)

    def error_word(self):
        return self.zeros(1, torch.int32)

    def check(self, what=""):
        torch.cuda.synchronize()
        for i, (buf, nbytes, head, tail) in enumerate(self.items):
            h = buf[:GUARD].cpu().numpy()
            tl = buf[GUARD + nbytes:].cpu().numpy()
            assert h.tobytes() == head.tobytes(), f"{what}: guard before array {i} overwritten"
            assert tl.tobytes() == tail.tobytes(), f"{what}: guard after array {i} overwritten"


# ---------------------------------------------------------------- planted specials
# fp32 bit patterns planted in coordinates no step touches: NaN payloads (quiet,
# negative, signalling), infinities, -0.0, denormals.
SPECIAL_BITS = np.array([0x7FC00001, 0xFFC12345, 0x7F800001, 0x7F800000, 0xFF800000, 0x80000000,
                         0x00000001, 0x807FFFFF, 0x00400000], dtype=np.uint32)


def plant_specials(arr, never_touched, rng, k=64):
    """Writes special values into up to k never-touched coordinates of arr (in place)."""
    flat = np.flatnonzero(np.asarray(never_touched).reshape(-1))
    if flat.size == 0:
        return
    pick = rng.choice(flat, min(k, flat.size), replace=False)
    arr.reshape(-1).view(np.uint32)[pick] = SPECIAL_BITS[rng.integers(0, SPECIAL_BITS.size, pick.size)]


def dev(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host(t):
    return t.detach().cpu().numpy()
