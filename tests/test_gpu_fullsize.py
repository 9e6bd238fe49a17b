"""Parity at the specified full sizes and step counts, on sampled rows.

Each 2-D workload runs at its full size, for its full number of steps, through the C-ABI
entry point bench.py times (the same launch configuration).  The oracle cannot redo a 15 GB
table, but every row's update depends only on that row's state and the gradient entries that
name it, so the oracle runs on a reduced table holding just the sampled rows, fed every
step's entries for those rows in their original input order (duplicates intact): its results
are exactly what the full oracle gives for those rows.  The GPU state of the sampled rows is
read back and compared after steps 1, 2, 10 and the last one: touched rows within the parity
tolerance (|x - r| <= max(1e-5 |r|, 1e-7)), second moments within 1e-5 relative with no
floor, first moments within 1e-5 of their magnitude scale (gpu_harness), last_step exact,
rows or coordinates not yet touched bit-identical to the initial table.  Sampled rows are
chosen before the run: the Zipf head (the longest duplicate segments), random rows of the
first step, random rows of the whole table (mostly never touched under Zipf).  Sampled
coordinates that no step touches hold planted specials (NaN payloads, infinities, -0.0,
denormals) in every state array, and every state array and the workspace sit inside guard
regions checked at each comparison.
"""
from __future__ import annotations

from collections import deque
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
from gpu_harness import (Guarded, MomentScale, SPECIAL_BITS, assert_m_scaled, assert_state_close, assert_v_relative,
                         dev, host)
from lazy_optimizers_embedding_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _checkpoints(steps):
    return sorted({s for s in (1, 2, 10, steps) if 1 <= s <= steps})


def _stream(make, steps, ahead=4):
    """make(0), make(1), ... in order, each drawn on a thread pool a few steps ahead."""
    with ThreadPoolExecutor(max_workers=ahead) as ex:
        q = deque(ex.submit(make, s) for s in range(min(ahead, steps)))
        for s in range(steps):
            out = q.popleft().result()
            if s + ahead < steps:
                q.append(ex.submit(make, s + ahead))
            yield out


def _pick_rows(w, first_touched, rng, hot=8, k_touched=96, k_random=32):
    parts = [np.arange(min(hot, w.rows), dtype=np.int64)] if w.index_dist == "zipf" else []
    parts.append(rng.choice(first_touched, min(k_touched, first_touched.shape[0]), replace=False))
    parts.append(rng.integers(0, w.rows, k_random, dtype=np.int64))
    return np.unique(np.concatenate(parts))


def _specials(rng, shape):
    """fp32 array of the given shape filled with planted special values."""
    return SPECIAL_BITS[rng.integers(0, SPECIAL_BITS.size, shape)].view(np.float32)


def _ever_touched_rows(w):
    """Every row any step of a row-COO workload lists."""
    with ThreadPoolExecutor(max_workers=8) as ex:
        parts = list(ex.map(lambda s: wl.step_indices(w, s), range(w.steps)))
    return np.unique(np.concatenate(parts))


def _free():
    import torch
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _raw_coo_full_run(so, w, dd=True):
    """Every step of a raw row-COO workload; compares the sampled rows at the checkpoints."""
    import torch
    key = f"{w.name}{'' if w.optimizer == 'sgd' else ('_dd' if dd else '_lazy')}"
    sgd = w.optimizer == "sgd"
    rows = _pick_rows(w, np.unique(wl.step_indices(w, 0)), np.random.default_rng(7))
    never = ~np.isin(rows, _ever_touched_rows(w))
    assert never.any()
    srng = np.random.default_rng(17)
    p0 = wl.table_init(w, threads=16)
    p0[rows[never]] = _specials(srng, (int(never.sum()), w.cols))
    G = Guarded(seed=3)
    p = G.array(p0)
    sel = torch.from_numpy(rows).cuda()
    sel_never = torch.from_numpy(rows[never]).cuda()
    err = G.error_word()
    ws = G.workspace(so, w.lookups, w.cols, w.rows)
    hp = p0[rows].copy()
    if sgd:
        buf = G.zeros((w.rows, w.cols))
        b0 = np.zeros_like(hp)
        b0[never] = _specials(srng, (int(never.sum()), w.cols))
        buf[sel_never] = dev(b0[never])
        hb = b0.copy()
        cfg = so.SgdConfig(lr=w.lr, momentum=w.momentum, weight_decay=w.weight_decay)
    else:
        m, v = G.zeros((w.rows, w.cols)), G.zeros((w.rows, w.cols))
        m0, v0 = np.zeros_like(hp), np.zeros_like(hp)
        m0[never] = _specials(srng, (int(never.sum()), w.cols))
        v0[never] = _specials(srng, (int(never.sum()), w.cols))
        m[sel_never], v[sel_never] = dev(m0[never]), dev(v0[never])
        ls = G.zeros(w.rows, torch.int64)
        hm, hv = m0.copy(), v0.copy()
        hls = np.zeros(rows.shape[0], np.int64)
        cfg = so.AdamConfig(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps)
        omode = oracle.MODE_DORMANCY_DECAY if dd else oracle.MODE_LAZY
        ohp = dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps)
        scale = MomentScale(hp.shape, rows.shape[0], ohp, omode, False)
    cps = _checkpoints(w.steps)
    touched = np.zeros(rows.shape[0], bool)
    checked = 0
    for t, (idx, vals) in enumerate(_stream(lambda s: wl.coo_step(w, s), w.steps), start=1):
        g = so.row_coo(dev(idx), dev(vals), False)
        if sgd:
            so.check(so.sparse_sgd_table_step(p, buf, w.rows, w.cols, g, cfg, ws, err), "sgd step")
        else:
            so.check(so.sparse_adam_table_step(p, m, v, ls, so.LAST_STEP_PER_ROW, w.rows, w.cols, g, t, cfg,
                                               so.DORMANCY_DECAY if dd else so.LAZY, ws, err), "adam step")
        keep = np.isin(idx, rows)
        ridx = np.searchsorted(rows, idx[keep]).astype(np.int64)   # rows is sorted and unique
        touched[np.unique(ridx)] = True
        if sgd:
            rc = oracle.sgd_table_step(hp, hb, lr=w.lr, momentum=w.momentum, weight_decay=w.weight_decay,
                                       rows=ridx, vals=vals[keep])
        else:
            scale.step(t, hp, rows=ridx, vals=vals[keep], is_canonical=False)
            rc = oracle.adam_table_step(hp, hm, hv, hls, t, mode=omode, rows=ridx, vals=vals[keep], **ohp)
        assert rc == 0
        if t in cps:
            torch.cuda.synchronize()
            assert int(err.item()) == 0, f"step {t}"
            G.check(f"step {t}")
            tmask = np.repeat(touched[:, None], w.cols, axis=1)
            assert_state_close(f"p@{t}", host(p[sel]), hp, tmask, p0[rows])
            if sgd:
                assert_state_close(f"buf@{t}", host(buf[sel]), hb, tmask, b0)
            else:
                gm, gv = host(m[sel]), host(v[sel])
                assert_state_close(f"m@{t}", gm, hm, tmask, m0)
                assert_state_close(f"v@{t}", gv, hv, tmask, v0)
                assert_v_relative(key, f"v@{t}", gv, hv, tmask)
                assert_m_scaled(key, f"m@{t}", gm, hm, scale.M, tmask)
                assert np.array_equal(host(ls[sel]), hls), f"last_step@{t}"
            checked += 1
    assert checked == len(cps)
    if w.index_dist == "zipf":
        assert touched[0] and (~touched).sum() > 5
    assert touched.sum() > 50
    del p, ws, G
    if sgd:
        del buf
    else:
        del m, v, ls
    _free()


@pytest.mark.parametrize("dd", [True, False], ids=["dormancy_decay", "lazy"])
def test_table_10Mx128_zipf_raw_coo_adam_fullsize(cuda_lib, dd):
    _raw_coo_full_run(cuda_lib, wl.CFG_ZIPF_10M_128, dd)


def test_table_50Mx32_uniform_raw_coo_sgd_fullsize(cuda_lib):
    _raw_coo_full_run(cuda_lib, wl.CFG_SGD_50M_32)


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


def _csr_touched_of_rows(make, steps, rows, cols):
    """Coordinates of the given rows that any step of a CSR workload lists."""
    mask = np.zeros((rows.shape[0], cols), bool)

    def one(s):
        ro, co, _ = make(s)
        so_off, so_cols, _ = _csr_rows_subset(ro, co, co, rows)
        return so_off, so_cols

    with ThreadPoolExecutor(max_workers=4) as ex:
        for so_off, so_cols in ex.map(one, range(steps)):
            rr = np.repeat(np.arange(rows.shape[0]), np.diff(so_off))
            mask[rr, so_cols] = True
    return mask


@pytest.mark.parametrize("cfg", ["1Mx64_zipf_csr_full_rows", "4Mx256_csr_element_per_coord"])
def test_csr_adam_fullsize(cuda_lib, cfg):
    import torch
    so = cuda_lib
    if cfg.startswith("1M"):
        w, per_coord = wl.CFG_ZIPF_1M_64, False
        make = lambda s: _summed_csr(w, s)   # noqa: E731
        first = np.unique(wl.step_indices(w, 0))
    else:
        w, per_coord = wl.CFG_CSR_4M_256, True
        make = lambda s: wl.csr_elem_step(w, s)   # noqa: E731
        first = wl.step_indices(w, 0)
    key = w.name
    rows = _pick_rows(w, first, np.random.default_rng(11))
    if per_coord:
        ever = _csr_touched_of_rows(make, w.steps, rows, w.cols)
    else:
        ever = np.repeat(np.isin(rows, _ever_touched_rows(w))[:, None], w.cols, axis=1)
    never = ~ever
    assert never.any()
    srng = np.random.default_rng(19)
    p0 = wl.table_init(w, threads=16)
    hp = p0[rows].copy()
    hp[never] = _specials(srng, int(never.sum()))
    p0[rows] = hp
    m0, v0 = np.zeros_like(hp), np.zeros_like(hp)
    m0[never] = _specials(srng, int(never.sum()))
    v0[never] = _specials(srng, int(never.sum()))
    G = Guarded(seed=5)
    p = G.array(p0)
    sel = torch.from_numpy(rows).cuda()
    m, v = G.zeros((w.rows, w.cols)), G.zeros((w.rows, w.cols))
    m[sel], v[sel] = dev(m0), dev(v0)
    ls = G.zeros(w.rows * w.cols if per_coord else w.rows, torch.int64)
    err = G.error_word()
    # the workspace the benchmark passes: full rows then take the row kernel, element entries the flat update
    ws = G.workspace(so, w.lookups * w.csr_cols_per_row + 64, 1, w.rows) if per_coord else \
        G.workspace(so, w.lookups + 1, 1, w.rows)
    cfgc = so.AdamConfig(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps)
    ohp = dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps)
    layout = so.LAST_STEP_PER_COORD if per_coord else so.LAST_STEP_PER_ROW
    cps = _checkpoints(w.steps)
    hm, hv = m0.copy(), v0.copy()
    hls = np.zeros(hp.size if per_coord else rows.shape[0], np.int64)
    scale = MomentScale(hp.shape, hls.shape[0], ohp, oracle.MODE_DORMANCY_DECAY, per_coord)
    tmask = np.zeros(hp.shape, bool)
    checked = 0
    for t, (ro, co, va) in enumerate(_stream(make, w.steps), start=1):
        g = so.csr(dev(ro), dev(co), dev(va))
        so.check(so.sparse_adam_table_step(p, m, v, ls, layout, w.rows, w.cols, g, t, cfgc, so.DORMANCY_DECAY,
                                           ws, err), "csr step")
        so_off, so_cols, so_vals = _csr_rows_subset(ro, co, va, rows)
        for i in range(rows.shape[0]):
            tmask[i, so_cols[so_off[i]:so_off[i + 1]]] = True
        scale.step(t, hp, row_off=so_off, cols=so_cols, vals=so_vals)
        rc = oracle.adam_table_step(hp, hm, hv, hls, t, mode=oracle.MODE_DORMANCY_DECAY, row_off=so_off,
                                    cols=so_cols, vals=so_vals, ls_per_coord=per_coord, **ohp)
        assert rc == 0
        if t in cps:
            torch.cuda.synchronize()
            assert int(err.item()) == 0, f"step {t}"
            G.check(f"step {t}")
            gm, gv = host(m[sel]), host(v[sel])
            assert_state_close(f"p@{t}", host(p[sel]), hp, tmask, p0[rows])
            assert_state_close(f"m@{t}", gm, hm, tmask, m0)
            assert_state_close(f"v@{t}", gv, hv, tmask, v0)
            assert_v_relative(key, f"v@{t}", gv, hv, tmask)
            assert_m_scaled(key, f"m@{t}", gm, hm, scale.M, tmask)
            got_ls = host(ls.view(w.rows, w.cols)[sel]) if per_coord else host(ls[sel])
            assert np.array_equal(got_ls.reshape(-1), hls.reshape(-1)), f"last_step@{t}"
            checked += 1
    assert checked == len(cps)
    assert tmask.any() and (~tmask).any()
    del p, m, v, ls, G
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
