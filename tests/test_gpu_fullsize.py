"""Parity at the specified full sizes, on sampled rows.

Each workload runs at its full size through the C-ABI entry point bench.py times (the same
launch configuration), for a few steps.  The oracle cannot redo a 15 GB table, but every row's
update depends only on that row's state and the gradient entries that name it, so the oracle
runs on a reduced table holding just the sampled rows, fed the same steps' entries for those
rows in their original input order (duplicates intact): its results are exactly what the full
oracle gives for those rows.  Checked per sampled row: touched rows within the parity
tolerance (|x - r| <= max(1e-5 |r|, 1e-7)), last_step exact, untouched rows bit-identical to
the initial table.  Samples: the hottest rows (Zipf head, the longest duplicate segments),
random touched rows, random untouched rows.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from gpu_harness import assert_state_close, dev, host
from lazy_optimizers_embedding_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

STEPS = 3


def _sample_rows(w, touched_sets, rng, hot=8, k_touched=96, k_untouched=32):
    touched = np.unique(np.concatenate(touched_sets))
    out = [touched[:hot]]                                    # lowest ids: the Zipf head
    out.append(rng.choice(touched, min(k_touched, touched.shape[0]), replace=False))
    mask = np.ones(w.rows, bool)
    mask[touched] = False
    untouched = np.flatnonzero(mask)
    out.append(rng.choice(untouched, min(k_untouched, untouched.shape[0]), replace=False))
    return np.unique(np.concatenate(out))


def _free():
    import torch
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _run_raw_coo(so, w, dd=True):
    """Raw row-COO steps of a full-size table; returns the sampled rows' GPU and oracle state."""
    import torch
    batches = [wl.coo_step(w, s) for s in range(STEPS)]
    p0 = wl.table_init(w, threads=16)
    p = dev(p0)
    sgd = w.optimizer == "sgd"
    err = so.error_word()
    ws = so.workspace(w.lookups, w.cols, w.rows)
    if sgd:
        buf = torch.zeros_like(p)
        cfg = so.SgdConfig(lr=w.lr, momentum=w.momentum, weight_decay=w.weight_decay)
    else:
        m, v = torch.zeros_like(p), torch.zeros_like(p)
        ls = torch.zeros(w.rows, dtype=torch.int64, device="cuda")
        cfg = so.AdamConfig(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps)
    for t, (idx, vals) in enumerate(batches, start=1):
        g = so.row_coo(dev(idx), dev(vals), False)
        if sgd:
            so.check(so.sparse_sgd_table_step(p, buf, w.rows, w.cols, g, cfg, ws, err), "sgd step")
        else:
            so.check(so.sparse_adam_table_step(p, m, v, ls, so.LAST_STEP_PER_ROW, w.rows, w.cols, g, t, cfg,
                                               so.DORMANCY_DECAY if dd else so.LAZY, ws, err), "adam step")
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = _sample_rows(w, [b[0] for b in batches], np.random.default_rng(7))
    sel = torch.from_numpy(rows).cuda()
    got = {"p": host(p[sel])}
    if sgd:
        got["buf"] = host(buf[sel])
    else:
        got.update(m=host(m[sel]), v=host(v[sel]), ls=host(ls[sel]))
    # the oracle on the reduced table
    hp = p0[rows].copy()
    ref = {}
    if sgd:
        hb = np.zeros_like(hp)
    else:
        hm, hv = np.zeros_like(hp), np.zeros_like(hp)
        hls = np.zeros(rows.shape[0], np.int64)
    for t, (idx, vals) in enumerate(batches, start=1):
        keep = np.isin(idx, rows)
        ridx = np.searchsorted(rows, idx[keep]).astype(np.int64)   # rows is sorted and unique
        rvals = vals[keep]
        if sgd:
            rc = oracle.sgd_table_step(hp, hb, lr=w.lr, momentum=w.momentum, weight_decay=w.weight_decay,
                                       rows=ridx, vals=rvals)
        else:
            rc = oracle.adam_table_step(hp, hm, hv, hls, t, lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps,
                                        mode=oracle.MODE_DORMANCY_DECAY if dd else oracle.MODE_LAZY,
                                        rows=ridx, vals=rvals)
        assert rc == 0
    ref["p"] = hp
    if sgd:
        ref["buf"] = hb
    else:
        ref.update(m=hm, v=hv, ls=hls)
    touched = np.isin(rows, np.unique(np.concatenate([b[0] for b in batches])))
    del p, ws
    if sgd:
        del buf
    else:
        del m, v, ls
    _free()
    return rows, touched, p0[rows], got, ref


@pytest.mark.parametrize("dd", [True, False], ids=["dormancy_decay", "lazy"])
def test_table_10Mx128_zipf_raw_coo_adam_fullsize(cuda_lib, dd):
    rows, touched, init, got, ref = _run_raw_coo(cuda_lib, wl.CFG_ZIPF_10M_128, dd)
    tmask = np.repeat(touched[:, None], wl.CFG_ZIPF_10M_128.cols, axis=1)
    for k in ("p", "m", "v"):
        assert_state_close(k, got[k], ref[k], tmask, init if k == "p" else np.zeros_like(init))
    assert np.array_equal(got["ls"], ref["ls"])
    assert touched[0] and touched.sum() > 50 and (~touched).sum() > 10


def test_table_50Mx32_uniform_raw_coo_sgd_fullsize(cuda_lib):
    w = wl.CFG_SGD_50M_32
    rows, touched, init, got, ref = _run_raw_coo(cuda_lib, w)
    tmask = np.repeat(touched[:, None], w.cols, axis=1)
    assert_state_close("p", got["p"], ref["p"], tmask, init)
    assert_state_close("buf", got["buf"], ref["buf"], tmask, np.zeros_like(init))


def _csr_rows_subset(row_off, cols, vals, rows):
    """The CSR of a full table restricted to `rows` (renumbered 0..len-1)."""
    counts = row_off[rows + 1] - row_off[rows]
    sub_off = np.zeros(rows.shape[0] + 1, np.int64)
    np.cumsum(counts, out=sub_off[1:])
    take = np.concatenate([np.arange(row_off[r], row_off[r + 1]) for r in rows]) if counts.sum() else \
        np.zeros(0, np.int64)
    return sub_off, cols[take], vals[take]


def _summed_csr(w, step):
    """A step of summed Zipf lookups as a full-row CSR (duplicates summed in fp64, rounded once)."""
    idx, vals = wl.coo_step(w, step)
    uidx, inv = np.unique(idx, return_inverse=True)
    s = np.zeros((uidx.shape[0], w.cols), np.float64)
    np.add.at(s, inv, vals.astype(np.float64))
    row_off = np.zeros(w.rows + 1, np.int64)
    cnt = np.zeros(w.rows, np.int64)
    cnt[uidx] = w.cols
    np.cumsum(cnt, out=row_off[1:])
    cols = np.tile(np.arange(w.cols, dtype=np.int32), uidx.shape[0])
    return row_off, cols, s.astype(np.float32).reshape(-1)


@pytest.mark.parametrize("cfg", ["1Mx64_zipf_csr_full_rows", "4Mx256_csr_element_per_coord"])
def test_csr_adam_fullsize(cuda_lib, cfg):
    import torch
    so = cuda_lib
    if cfg.startswith("1M"):
        w, per_coord = wl.CFG_ZIPF_1M_64, False
        steps = [_summed_csr(w, s) for s in range(STEPS)]
    else:
        w, per_coord = wl.CFG_CSR_4M_256, True
        steps = [wl.csr_elem_step(w, s) for s in range(STEPS)]
    p0 = wl.table_init(w, threads=16)
    p = dev(p0)
    m, v = torch.zeros_like(p), torch.zeros_like(p)
    ls = torch.zeros(w.rows * w.cols if per_coord else w.rows, dtype=torch.int64, device="cuda")
    err = so.error_word()
    cfgc = so.AdamConfig(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps)
    layout = so.LAST_STEP_PER_COORD if per_coord else so.LAST_STEP_PER_ROW
    for t, (ro, co, va) in enumerate(steps, start=1):
        g = so.csr(dev(ro), dev(co), dev(va))
        so.check(so.sparse_adam_table_step(p, m, v, ls, layout, w.rows, w.cols, g, t, cfgc, so.DORMANCY_DECAY,
                                           None, err), "csr step")
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    touched_sets = [np.flatnonzero(np.diff(ro)) for ro, _, _ in steps]
    rows = _sample_rows(w, touched_sets, np.random.default_rng(11))
    sel = torch.from_numpy(rows).cuda()
    got_p, got_m, got_v = host(p[sel]), host(m[sel]), host(v[sel])
    got_ls = host(ls.view(w.rows, w.cols)[sel]) if per_coord else host(ls[sel])
    hp = p0[rows].copy()
    hm, hv = np.zeros_like(hp), np.zeros_like(hp)
    hls = np.zeros(hp.size if per_coord else rows.shape[0], np.int64)
    tmask = np.zeros(hp.shape, bool)
    for t, (ro, co, va) in enumerate(steps, start=1):
        so_off, so_cols, so_vals = _csr_rows_subset(ro, co, va, rows)
        for i in range(rows.shape[0]):
            tmask[i, so_cols[so_off[i]:so_off[i + 1]]] = True
        rc = oracle.adam_table_step(hp, hm, hv, hls, t, lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps,
                                    mode=oracle.MODE_DORMANCY_DECAY, row_off=so_off, cols=so_cols, vals=so_vals,
                                    ls_per_coord=per_coord)
        assert rc == 0
    assert_state_close("p", got_p, hp, tmask, p0[rows])
    assert_state_close("m", got_m, hm, tmask, np.zeros_like(hp))
    assert_state_close("v", got_v, hv, tmask, np.zeros_like(hp))
    assert np.array_equal(got_ls.reshape(-1), hls.reshape(-1))
    assert tmask.any() and (~tmask).any()
    del p, m, v, ls
    _free()


def test_read_rows_10Mx128_zipf_fullsize(cuda_lib):
    """The forward gather of the 10M x 128 table at one step's 262,144 Zipf lookups, bit for bit."""
    import torch
    so = cuda_lib
    w = wl.CFG_ZIPF_10M_128
    p0 = wl.table_init(w, threads=16)
    idx = wl.step_indices(w, 0)
    out = torch.empty((idx.shape[0], w.cols), dtype=torch.float32, device="cuda")
    err = so.error_word()
    t = dev(p0)
    so.check(so.sparse_read_rows(t, w.rows, w.cols, dev(idx), idx.shape[0], out, err), "read_rows")
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert host(out).tobytes() == oracle.read_rows(p0, idx).tobytes()
    del t, out
    _free()
