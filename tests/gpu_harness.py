"""Shared helpers of the GPU parity tests: run a step sequence through the C-ABI
(binding) and the same sequence through the CPU oracle, then compare.

Tolerance for fp32 state (p, m, v, buf): |gpu - ref| <= max(1e-5 |ref|, 1e-7)
for every coordinate; untouched coordinates bitwise; last_step exactly.
"""
from __future__ import annotations

import numpy as np
import torch

RTOL = 1e-5
ATOL = 1e-7


def tol_violations(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    g = got.astype(np.float64)
    r = ref.astype(np.float64)
    bad = ~(np.abs(g - r) <= np.maximum(RTOL * np.abs(r), ATOL))
    both_nan = np.isnan(g) & np.isnan(r)
    return bad & ~both_nan


def assert_state_close(name, got, ref, touched_mask=None, init=None):
    got = np.asarray(got)
    ref = np.asarray(ref)
    bad = tol_violations(got, ref)
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} outside tolerance; first {i.tolist()}: "
                             f"gpu {got[tuple(i.T)]} ref {ref[tuple(i.T)]}")
    if touched_mask is not None and init is not None:
        un = ~touched_mask
        assert got[un].tobytes() == np.asarray(init)[un].tobytes(), f"{name}: untouched coordinates changed"


def max_rel(got, ref):
    g = np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    nz = r != 0
    return float(np.max(np.abs(g[nz] - r[nz]) / np.abs(r[nz]))) if nz.any() else 0.0


def dev(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host(t):
    return t.detach().cpu().numpy()
