"""sparse_canonicalize_static_ws: canonicalisation for callers that cannot allocate.

Some callers of this library cannot obtain device memory for a workspace (a
host application that owns every device allocation through its own pool, or a
thread where cudaMalloc is not allowed).  This entry point runs the same kernels
as sparse_canonicalize but takes its scratch from a fixed device array compiled
into the library.  These tests call it through the C ABI twice in a row, on
inputs of different shapes (so the second call starts from the first call's
leftovers in the shared array), and check every output against
sparse_canonicalize with an ordinary caller workspace: indices, run boundaries
and the permutation bit for bit, summed values within the parity tolerance.
The file is named so that pytest collects it last.
"""
import numpy as np
import pytest

from gpu_harness import dev, host, tol_violations

pytestmark = pytest.mark.gpu


def _outputs(torch, n, c):
    return (torch.empty(n, dtype=torch.int64, device="cuda"),
            torch.empty((n, c), dtype=torch.float32, device="cuda"),
            torch.empty(n + 1, dtype=torch.int64, device="cuda"),
            torch.empty(n, dtype=torch.int64, device="cuda"),
            torch.full((1,), -1, dtype=torch.int64, device="cuda"))


def _canonicalize_both(so, torch, idx, vals, bound):
    n, c = vals.shape
    d_idx, d_vals = dev(idx), dev(vals)
    ref = _outputs(torch, n, c)
    got = _outputs(torch, n, c)
    err_ref, err_got = so.error_word(), so.error_word()
    so.check(so.sparse_canonicalize(d_idx, d_vals, n, c, bound, *ref, so.workspace(n, c, bound), err_ref),
             "sparse_canonicalize")
    so.check(so.sparse_canonicalize_static_ws(d_idx, d_vals, n, c, bound, *got, err_got),
             "sparse_canonicalize_static_ws")
    torch.cuda.synchronize()
    assert int(err_ref.item()) == 0 and int(err_got.item()) == 0
    u = int(ref[4].item())
    assert int(got[4].item()) == u
    assert np.array_equal(host(got[0])[:u], host(ref[0])[:u])
    assert np.array_equal(host(got[2])[:u + 1], host(ref[2])[:u + 1])
    assert np.array_equal(host(got[3]), host(ref[3]))
    gv, rv = host(got[1])[:u], host(ref[1])[:u]
    assert not tol_violations(gv, rv).any()
    return u


def test_static_workspace_matches_caller_workspace_two_calls(cuda_lib):
    so = cuda_lib
    import torch
    rng = np.random.default_rng(20)
    # call 1: many duplicates of one hot key (multi-level combining tree), 64 columns
    n1, c1, b1 = 50_000, 64, 20_000
    idx1 = rng.integers(0, b1, n1).astype(np.int64)
    idx1[rng.choice(n1, 6000, replace=False)] = 7
    vals1 = rng.standard_normal((n1, c1)).astype(np.float32)
    u1 = _canonicalize_both(so, torch, idx1, vals1, b1)
    # call 2: a smaller input of another shape reuses the same array right after
    n2, c2, b2 = 3_001, 128, 900
    idx2 = rng.integers(0, b2, n2).astype(np.int64)
    vals2 = rng.standard_normal((n2, c2)).astype(np.float32)
    u2 = _canonicalize_both(so, torch, idx2, vals2, b2)
    assert 0 < u1 <= n1 and 0 < u2 <= n2


def test_static_workspace_rejects_sizes_beyond_its_limit(cuda_lib):
    so = cuda_lib
    import torch
    n, c, bound = 200_000, 256, 1_000_000
    assert so.sparse_workspace_size(n, c, bound) > so.STATIC_WS_BYTES
    idx = torch.zeros(n, dtype=torch.int64, device="cuda")
    vals = torch.zeros((n, c), dtype=torch.float32, device="cuda")
    outs = _outputs(torch, n, c)
    err = so.error_word()
    assert so.sparse_canonicalize_static_ws(idx, vals, n, c, bound, *outs, err) == so.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(outs[4].item()) == -1 and int(err.item()) == 0  # nothing was enqueued


def _largest_n(so, c, bound):
    """The largest entry count whose workspace fits the static array (workspace size grows with n)."""
    lo, hi = 1, 1 << 24
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if so.sparse_workspace_size(mid, c, bound) <= so.STATIC_WS_BYTES:
            lo = mid
        else:
            hi = mid - 1
    return lo


def test_static_workspace_size_boundary(cuda_lib):
    """The largest call that fits the array is accepted and correct; one entry more is refused."""
    so = cuda_lib
    import torch
    c, bound = 256, 1_000_000
    n = _largest_n(so, c, bound)
    assert so.sparse_workspace_size(n + 1, c, bound) > so.STATIC_WS_BYTES
    rng = np.random.default_rng(21)
    idx = rng.integers(0, bound, n).astype(np.int64)
    idx[:2000] = 3
    vals = rng.standard_normal((n, c)).astype(np.float32)
    _canonicalize_both(so, torch, idx, vals, bound)
    d_idx, d_vals = dev(np.zeros(n + 1, np.int64)), dev(np.zeros((n + 1, c), np.float32))
    outs = _outputs(torch, n + 1, c)
    err = so.error_word()
    assert so.sparse_canonicalize_static_ws(d_idx, d_vals, n + 1, c, bound, *outs, err) == so.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(outs[4].item()) == -1 and int(err.item()) == 0


def test_static_workspace_allocates_nothing(cuda_lib):
    """After the first call on the device (which may load the library's device code and so create
    the array), further calls leave the device's free memory unchanged."""
    so = cuda_lib
    import torch
    rng = np.random.default_rng(22)
    n, c, bound = 40_000, 32, 5_000
    d_idx = dev(rng.integers(0, bound, n).astype(np.int64))
    d_vals = dev(rng.standard_normal((n, c)).astype(np.float32))
    outs = _outputs(torch, n, c)
    err = so.error_word()
    so.check(so.sparse_canonicalize_static_ws(d_idx, d_vals, n, c, bound, *outs, err), "first call")
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        so.check(so.sparse_canonicalize_static_ws(d_idx, d_vals, n, c, bound, *outs, err), "later call")
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert int(err.item()) == 0 and int(outs[4].item()) > 0
