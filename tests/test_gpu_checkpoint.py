"""Save and resume: optimizer state saved to the host in the middle of a run, restored into
fresh device arrays, continues bit for bit like the uninterrupted run.

The library keeps no state between calls, so everything a run needs to continue is the
caller's: p, m, v and last_step (Adam) or p and the momentum buffer (SGD), plus the global
step t.  ("DiskSparseAdam (DSA)" README, "Portable Checkpoints": a checkpoint restores the
weights, moments, per-row counters and the global step; the disk format itself is out of
scope here.)  Every addition order is fixed, so the continuation must match exactly.
"""
import numpy as np
import pytest

from gpu_harness import dev, host
from lazy_optimizers_embedding_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _adam_steps(so, w, state, t0, t1, mode, ws, err):
    p, m, v, ls = state
    cfg = so.AdamConfig(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps)
    for t in range(t0, t1 + 1):
        idx, vals = wl.coo_step(w, t - 1)
        so.check(so.sparse_adam_table_step(p, m, v, ls, so.LAST_STEP_PER_ROW, w.rows, w.cols,
                                           so.row_coo(dev(idx), dev(vals), False), t, cfg, mode, ws, err))


@pytest.mark.parametrize("mode", [0, 1], ids=["lazy", "dormancy_decay"])
def test_adam_resume_is_bit_identical(cuda_lib, mode):
    import torch
    so = cuda_lib
    w = wl.CFG_ZIPF_10M_128.scaled(rows=40_000, cols=64, lookups=20_000, steps=9)
    p0 = wl.table_init(w)
    err = so.error_word()
    ws = so.workspace(w.lookups, w.cols, w.rows)
    full = (dev(p0), torch.zeros((w.rows, w.cols), device="cuda"), torch.zeros((w.rows, w.cols), device="cuda"),
            torch.zeros(w.rows, dtype=torch.int64, device="cuda"))
    k = 4
    _adam_steps(so, w, full, 1, k, mode, ws, err)
    torch.cuda.synchronize()
    saved = [host(a).copy() for a in full]   # the checkpoint, with t = k
    _adam_steps(so, w, full, k + 1, w.steps, mode, ws, err)
    resumed = tuple(dev(a) for a in saved)
    ws2, err2 = so.workspace(w.lookups, w.cols, w.rows), so.error_word()
    _adam_steps(so, w, resumed, k + 1, w.steps, mode, ws2, err2)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and int(err2.item()) == 0
    for name, a, b in zip(("p", "m", "v", "last_step"), full, resumed):
        assert host(a).tobytes() == host(b).tobytes(), f"{name} differs after resuming"
    assert not np.array_equal(saved[0], host(full[0])), "the continuation changed nothing"


def test_sgd_resume_is_bit_identical(cuda_lib):
    import torch
    so = cuda_lib
    w = wl.CFG_SGD_50M_32.scaled(rows=60_000, lookups=30_000, steps=7)
    p0 = wl.table_init(w)
    cfg = so.SgdConfig(lr=w.lr, momentum=w.momentum, weight_decay=w.weight_decay)
    err = so.error_word()

    def run(p, buf, t0, t1, ws):
        for t in range(t0, t1 + 1):
            idx, vals = wl.coo_step(w, t - 1)
            so.check(so.sparse_sgd_table_step(p, buf, w.rows, w.cols, so.row_coo(dev(idx), dev(vals), False), cfg,
                                              ws, err))

    p, buf = dev(p0), torch.zeros((w.rows, w.cols), device="cuda")
    k = 3
    run(p, buf, 1, k, so.workspace(w.lookups, w.cols, w.rows))
    torch.cuda.synchronize()
    saved = (host(p).copy(), host(buf).copy())
    run(p, buf, k + 1, w.steps, so.workspace(w.lookups, w.cols, w.rows))
    rp, rb = dev(saved[0]), dev(saved[1])
    run(rp, rb, k + 1, w.steps, so.workspace(w.lookups, w.cols, w.rows))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert host(p).tobytes() == host(rp).tobytes() and host(buf).tobytes() == host(rb).tobytes()
