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
