"""GPU path (through the C-ABI) against the CPU oracle, element by element.

Sizes: the oracle finishes each case in well under a second, while the inputs
still span several radix / run-detection tiles (2,048 entries each), several
pieces of 32 sorted entries, a ragged tail, and hot keys with enough duplicates
to need two levels of the partial-combining tree (> 32*32 entries of one key).
"""
import os

import numpy as np
import pytest

import oracle
from gpu_harness import (Guarded, MomentScale, assert_m_scaled, assert_state_close, assert_v_relative, dev, host,
                         max_rel, plant_specials, tol_violations)

pytestmark = pytest.mark.gpu

ADAM = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)


def _raw_rows(rng, n, bound, hot=None, hot_count=0):
    idx = rng.integers(0, bound, n).astype(np.int64)
    if hot is not None and hot_count:
        pos = rng.choice(n, size=min(hot_count, n), replace=False)
        idx[pos] = hot
    return idx


# ------------------------------------------------------------------ canonicalize
CANON_CASES = [
    # (n, c, bound, hot_count)
    (1, 1, 1, 0),
    (7, 3, 10, 0),
    (2048, 4, 1000, 0),
    (5000, 1, 10_000_000, 0),
    (5000, 32, 1000, 1500),
    (9000, 64, 4000, 3000),
    (20000, 128, 50_000, 4500),
    (3001, 256, 50, 0),
    (1500, 1000, 300, 200),
    (4096, 5, 1, 0),          # every entry the same key
    (70_000, 2, 100_000, 0),
    (600_000, 1, 2_000_000, 3000),   # large-input tiles (16 keys per thread), 21-bit keys
    (530_000, 4, 40_000_000, 0),     # large-input tiles, 26-bit keys (four passes)
    (5000, 2, 2**32, 300),           # 32-bit keys at the bound's cap, hot key 2^32 - 1 (all bits set)
    (3000, 1, 2**31 + 7, 0),         # keys above 2^31
]


@pytest.mark.parametrize("n,c,bound,hot", CANON_CASES)
def test_canonicalize_matches_oracle(cuda_lib, n, c, bound, hot):
    so = cuda_lib
    import torch
    rng = np.random.default_rng(n * 7 + c)
    idx = _raw_rows(rng, n, bound, hot=bound - 1, hot_count=hot)
    vals = rng.standard_normal((n, c)).astype(np.float32)
    vals[rng.integers(0, n, max(1, n // 50))] = -0.0
    ri, rv, rseg, rperm = oracle.canonicalize(idx, vals, bound)
    u = ri.shape[0]
    G = Guarded(seed=n + c)
    d_idx = G.array(idx)
    d_vals = G.array(vals)
    idx_out = G.empty(n, torch.int64)
    vals_out = G.empty((n, c), torch.float32)
    seg_out = G.empty(n + 1, torch.int64)
    perm_out = G.empty(n, torch.int64)
    nnz = G.zeros(1, torch.int64)
    ws = G.workspace(so, n, c, bound)
    err = G.error_word()
    so.check(so.sparse_canonicalize(d_idx, d_vals, n, c, bound, idx_out, vals_out, seg_out, perm_out, nnz, ws,
                                    err), "canonicalize")
    G.check("canonicalize")
    assert host(d_idx).tobytes() == idx.tobytes() and host(d_vals).tobytes() == vals.tobytes(), "inputs changed"
    assert int(err.item()) == 0
    assert int(nnz.item()) == u
    assert np.array_equal(host(idx_out)[:u], ri)
    assert np.array_equal(host(seg_out)[:u + 1], rseg)
    assert np.array_equal(host(perm_out), rperm)
    gv = host(vals_out)[:u].reshape(u, c)
    rv = rv.reshape(u, c)
    bad = tol_violations(gv, rv)
    assert not bad.any(), f"{int(bad.sum())} values outside tolerance, max rel {max_rel(gv, rv)}"
    single = np.diff(rseg) == 1
    assert gv[single].tobytes() == rv[single].tobytes(), "a lone value must pass through bit for bit"


def test_canonicalize_empty_and_deterministic(cuda_lib):
    so = cuda_lib
    import torch
    err = so.error_word()
    nnz = torch.full((1,), 7, dtype=torch.int64, device="cuda")
    seg = torch.full((1,), 7, dtype=torch.int64, device="cuda")
    e = torch.empty(0, dtype=torch.int64, device="cuda")
    so.check(so.sparse_canonicalize(e, torch.empty(0, device="cuda"), 0, 4, 10, e, None, seg, None, nnz, None, err))
    torch.cuda.synchronize()
    assert int(nnz.item()) == 0 and int(seg.item()) == 0
    # keys are 32-bit: a bound above 2^32 is refused on the host, before anything is enqueued
    one = torch.zeros(1, dtype=torch.int64, device="cuda")
    assert so.sparse_canonicalize(one, torch.zeros(1, device="cuda"), 1, 1, 2**32 + 1, one, None, None, None, nnz,
                                  so.workspace(1, 1, 2**32), err) == so.ERR_INVALID_ARG
    rng = np.random.default_rng(3)
    n, c, bound = 30000, 64, 2000
    idx = _raw_rows(rng, n, bound, hot=5, hot_count=9000)
    vals = rng.standard_normal((n, c)).astype(np.float32)
    d_idx, d_vals = dev(idx), dev(vals)
    outs = []
    for _ in range(2):
        vo = torch.empty((n, c), device="cuda")
        io = torch.empty(n, dtype=torch.int64, device="cuda")
        so.check(so.sparse_canonicalize(d_idx, d_vals, n, c, bound, io, vo, None, None, nnz,
                                        so.workspace(n, c, bound), err))
        torch.cuda.synchronize()
        u = int(nnz.item())
        outs.append((u, host(io)[:u], host(vo)[:u]))
    assert int(err.item()) == 0
    assert outs[0][0] == outs[1][0]
    assert np.array_equal(outs[0][1], outs[1][1]) and outs[0][2].tobytes() == outs[1][2].tobytes()


# ------------------------------------------------------------------ lazy Adam, raw row-COO
def _test_key():
    return os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0].split("::")[-1]


def _run_adam(so, R, c, steps, mode, gen, form, layout=None, hp=ADAM, check_every=False, csr_ws=False):
    """gen(step) -> gradient for the step, in the given form; runs GPU and oracle side by side.

    Every device array is guarded (canaries checked after each step); coordinates that no step
    touches hold planted specials in p, m, v (and large or negative values in last_step) and
    must come back bit for bit; touched m and v are held to the no-floor checks of gpu_harness.
    csr_ws: CSR steps get a workspace (full rows with a per-row last_step then take the row path)."""
    import torch
    key = _test_key()
    rng = np.random.default_rng(R + c)
    grads = [gen(s) for s in range(steps)]
    per_coord = layout == so.LAST_STEP_PER_COORD
    ls_n = R * c if per_coord else R
    ever = np.zeros((R, c), bool)
    for g in grads:
        if form in ("raw", "canon"):
            ever[np.unique(g[0])] = True
        else:
            ever[np.repeat(np.arange(R), np.diff(g[0])), g[1]] = True
    p0 = (rng.standard_normal((R, c)) * 0.01).astype(np.float32)
    m0, v0 = np.zeros_like(p0), np.zeros_like(p0)
    srng = np.random.default_rng(99)
    for a in (p0, m0, v0):
        plant_specials(a, ~ever, srng)
    ls0 = np.zeros(ls_n, np.int64)
    ls_never = ~ever.reshape(-1) if per_coord else ~ever.any(axis=1)
    pick = np.flatnonzero(ls_never)[:16]
    ls0[pick] = np.where(np.arange(pick.size) % 2 == 0, np.int64(1) << 40, -5)
    G = Guarded(seed=R * 7 + c)
    p, m, v, ls = G.array(p0), G.array(m0), G.array(v0), G.array(ls0)
    op, om, ov, ols = p0.copy(), m0.copy(), v0.copy(), ls0.copy()
    err = G.error_word()
    cfg = so.AdamConfig(**hp)
    ohp = dict(hp)   # the oracle names the weight-decay mode wd_mode
    if "weight_decay_mode" in ohp:
        ohp["wd_mode"] = ohp.pop("weight_decay_mode")
    omode = oracle.MODE_DORMANCY_DECAY if mode == so.DORMANCY_DECAY else oracle.MODE_LAZY
    scale = MomentScale((R, c), ls_n, ohp, omode, per_coord)
    touched = np.zeros((R, c), bool)
    ws = None
    if form == "csr" and csr_ws:
        ws = G.workspace(so, max(g[1].shape[0] for g in grads) + 64, 1, R)
    for s in range(steps):
        t = s + 1
        g = grads[s]
        p_before = op.copy()
        if form == "raw" or form == "canon":
            rows, vals = g
            if ws is None and form == "raw":
                ws = G.workspace(so, max(rows.shape[0], 1), c, R)
            grad = so.row_coo(G.array(rows), G.array(vals), form == "canon")
            so.check(so.sparse_adam_table_step(p, m, v, ls, layout or so.LAST_STEP_PER_ROW, R, c, grad, t, cfg, mode,
                                               ws, err), "adam_table_step")
            rc = oracle.adam_table_step(op, om, ov, ols, t, rows=rows, vals=vals, is_canonical=(form == "canon"),
                                        mode=omode, ls_per_coord=per_coord, **ohp)
            scale.step(t, p_before, rows=rows, vals=vals, is_canonical=(form == "canon"))
            touched[np.unique(rows)] = True
        else:
            row_off, cols, vals = g
            grad = so.csr(G.array(row_off), G.array(cols), G.array(vals))
            so.check(so.sparse_adam_table_step(p, m, v, ls, layout, R, c, grad, t, cfg, mode, ws, err),
                     "adam_table_step csr")
            rc = oracle.adam_table_step(op, om, ov, ols, t, row_off=row_off, cols=cols, vals=vals, mode=omode,
                                        ls_per_coord=per_coord, **ohp)
            scale.step(t, p_before, row_off=row_off, cols=cols, vals=vals)
            rr = np.repeat(np.arange(R), np.diff(row_off))
            touched[rr, cols] = True
        assert rc == 0
        G.check(f"step {t}")
        assert int(err.item()) == 0, so.status_string(int(err.item()))
        if check_every or s == steps - 1:
            assert_state_close(f"p@t={t}", host(p), op, touched, p0)
            assert_state_close(f"m@t={t}", host(m), om, touched, m0)
            assert_state_close(f"v@t={t}", host(v), ov, touched, v0)
            assert_v_relative(key, f"v@t={t}", host(v), ov, touched)
            assert_m_scaled(key, f"m@t={t}", host(m), om, scale.M, touched)
            assert np.array_equal(host(ls), ols), f"last_step@t={t}"
    return host(p), host(m), host(v)


RAW_CASES = [(1, 1), (3, 3), (2000, 4), (3000, 32), (3000, 64), (2500, 128), (800, 256), (300, 1000)]


@pytest.mark.parametrize("mode", [0, 1], ids=["lazy", "dormancy_decay"])
@pytest.mark.parametrize("R,c", RAW_CASES)
def test_adam_raw_rows(cuda_lib, mode, R, c):
    so = cuda_lib

    def gen(s):
        rng = np.random.default_rng(1000 + s)
        n = 4000 if R > 3 else 50
        rows = _raw_rows(rng, n, R, hot=R // 2, hot_count=(1500 if s % 2 == 0 else 0) if R > 3 else 0)
        if R > 3:  # dormant rows: touch only part of the table per step
            rows = rows % max(1, R // (1 + s % 3))
        return rows, (rng.standard_normal((n, c)) * 0.01).astype(np.float32)

    _run_adam(so, R, c, 5, mode, gen, "raw", check_every=True)


@pytest.mark.parametrize("mode", [0, 1], ids=["lazy", "dormancy_decay"])
@pytest.mark.parametrize("R,c", [(5000, 1), (4000, 64), (3000, 128), (1000, 12)])
def test_adam_canonical_rows(cuda_lib, mode, R, c):
    so = cuda_lib

    def gen(s):
        rng = np.random.default_rng(2000 + s)
        rows = np.sort(rng.choice(R, size=R // 3, replace=False)).astype(np.int64)
        return rows, rng.standard_normal((rows.shape[0], c)).astype(np.float32)

    _run_adam(so, R, c, 4, mode, gen, "canon", check_every=True)


@pytest.mark.parametrize("mode", [0, 1], ids=["lazy", "dormancy_decay"])
def test_adam_raw_rows_per_coord_last_step(cuda_lib, mode):
    so = cuda_lib

    def gen(s):
        rng = np.random.default_rng(3000 + s)
        rows = _raw_rows(rng, 3000, 900, hot=3, hot_count=1200)
        return rows, rng.standard_normal((3000, 16)).astype(np.float32)

    _run_adam(so, 900, 16, 4, mode, gen, "raw", layout=so.LAST_STEP_PER_COORD)


def _csr_elem(rng, R, c, nrows, k):
    rows = np.sort(rng.choice(R, size=nrows, replace=False))
    counts = np.zeros(R, np.int64)
    counts[rows] = k
    row_off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    cols = np.sort(np.argsort(rng.random((nrows, c)), axis=1)[:, :k], axis=1).astype(np.int32).reshape(-1)
    return row_off, cols, rng.standard_normal(cols.shape[0]).astype(np.float32)


@pytest.mark.parametrize("csr_ws", [False, True], ids=["csr_kernel", "flat"])
@pytest.mark.parametrize("mode", [0, 1], ids=["lazy", "dormancy_decay"])
@pytest.mark.parametrize("R,c,nrows,k", [(2000, 256, 300, 16), (5000, 7, 1200, 3), (64, 40, 64, 40)])
def test_adam_csr_element_granular(cuda_lib, mode, R, c, nrows, k, csr_ws):
    """Element-granular CSR with a per-coordinate last_step, through the CSR kernel (no workspace) and
    through the flat one-entry-per-thread update (workspace given; the check records rows and gaps)."""
    so = cuda_lib
    _run_adam(so, R, c, 5, mode, lambda s: _csr_elem(np.random.default_rng(4000 + s), R, c, nrows, k), "csr",
              layout=so.LAST_STEP_PER_COORD, check_every=True, csr_ws=csr_ws)


@pytest.mark.parametrize("csr_ws", [False, True], ids=["csr_kernel", "row_path"])
@pytest.mark.parametrize("mode", [0, 1], ids=["lazy", "dormancy_decay"])
def test_adam_csr_full_rows_per_row_last_step(cuda_lib, mode, csr_ws):
    """A CSR whose listed rows are full, with one last_step per row (the summed-lookups shape), through the
    CSR kernel (no workspace) and through the row kernel over the compacted rows (workspace given)."""
    so = cuda_lib
    R, c = 3000, 64

    def gen(s):
        rng = np.random.default_rng(5000 + s)
        rows = np.sort(rng.choice(R, size=700, replace=False))
        ro, co = oracle.row_coo_to_csr(rows, R, c)
        return ro, co, rng.standard_normal(rows.shape[0] * c).astype(np.float32)

    _run_adam(so, R, c, 5, mode, gen, "csr", layout=so.LAST_STEP_PER_ROW, check_every=True, csr_ws=csr_ws)


@pytest.mark.parametrize("wd_mode", [0, 1], ids=["l2", "decoupled"])
@pytest.mark.parametrize("mode", [0, 1], ids=["lazy", "dormancy_decay"])
@pytest.mark.parametrize("form", ["raw", "canon", "csr_elem", "csr_full"])
def test_adam_weight_decay(cuda_lib, wd_mode, mode, form):
    """DSA's weight-decay modes on every gradient form, touched coordinates only."""
    so = cuda_lib
    hp = dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.05, weight_decay_mode=wd_mode)
    R, c = 3000, 64

    def gen(s):
        rng = np.random.default_rng(7000 + s)
        if form == "raw":
            rows = _raw_rows(rng, 2500, R, hot=5, hot_count=900) % max(1, R // (1 + s % 2))
            return rows, (rng.standard_normal((rows.shape[0], c)) * 0.01).astype(np.float32)
        if form == "canon":
            rows = np.sort(rng.choice(R, size=R // 4, replace=False)).astype(np.int64)
            return rows, rng.standard_normal((rows.shape[0], c)).astype(np.float32)
        if form == "csr_elem":
            return _csr_elem(rng, R, c, 400, 9)
        rows = np.sort(rng.choice(R, size=500, replace=False))
        ro, co = oracle.row_coo_to_csr(rows, R, c)
        return ro, co, rng.standard_normal(rows.shape[0] * c).astype(np.float32)

    f = "csr" if form.startswith("csr") else form
    layout = so.LAST_STEP_PER_COORD if form == "csr_elem" else so.LAST_STEP_PER_ROW
    _run_adam(so, R, c, 4, mode, gen, f, layout=layout, hp=hp, check_every=True, csr_ws=form.startswith("csr"))


def test_adam_weight_decay_bad_settings_rejected(cuda_lib):
    import torch
    so = cuda_lib
    p = torch.zeros((4, 4), device="cuda")
    m, v = torch.zeros_like(p), torch.zeros_like(p)
    ls = torch.zeros(4, dtype=torch.int64, device="cuda")
    g = so.row_coo(dev(np.array([1], np.int64)), dev(np.ones((1, 4), np.float32)), True)
    err = so.error_word()
    for kw in (dict(weight_decay=-0.1), dict(weight_decay=float("nan")), dict(weight_decay=0.1, weight_decay_mode=5)):
        cfg = so.AdamConfig(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, **kw)
        assert so.sparse_adam_table_step(p, m, v, ls, so.LAST_STEP_PER_ROW, 4, 4, g, 1, cfg, so.DORMANCY_DECAY,
                                         None, err) == so.ERR_INVALID_ARG


def test_summed_lookups_to_csr_then_step(cuda_lib):
    """Raw Zipf lookups -> GPU canonicalise -> GPU row-COO to CSR -> GPU CSR step, against the
    oracle's own canonicalise -> CSR -> step (each side from the same raw lookups)."""
    so = cuda_lib
    import torch
    from lazy_optimizers_embedding_gb300 import workloads as wl
    w = wl.CFG_ZIPF_1M_64.scaled(rows=20_000, lookups=6000, steps=4)
    R, c = w.rows, w.cols
    p0 = wl.table_init(w)
    p, m, v = dev(p0), torch.zeros((R, c), device="cuda"), torch.zeros((R, c), device="cuda")
    ls = torch.zeros(R, dtype=torch.int64, device="cuda")
    op, om, ov, ols = p0.copy(), np.zeros_like(p0), np.zeros_like(p0), np.zeros(R, np.int64)
    err = so.error_word()
    cfg = so.AdamConfig(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps)
    ws = so.workspace(w.lookups, c, R)
    for s in range(w.steps):
        t = s + 1
        idx, vals = wl.coo_step(w, s)
        n = idx.shape[0]
        d_idx, d_vals = dev(idx), dev(vals)
        io = torch.empty(n, dtype=torch.int64, device="cuda")
        vo = torch.empty((n, c), device="cuda")
        nnz = torch.zeros(1, dtype=torch.int64, device="cuda")
        so.check(so.sparse_canonicalize(d_idx, d_vals, n, c, R, io, vo, None, None, nnz, ws, err))
        torch.cuda.synchronize()
        u = int(nnz.item())
        ro = torch.empty(R + 1, dtype=torch.int64, device="cuda")
        co = torch.empty(max(u * c, 1), dtype=torch.int32, device="cuda")
        so.check(so.sparse_row_coo_to_csr(io, u, R, c, ro, co, err))
        vals_csr = vo[:u].contiguous().view(-1)
        so.check(so.sparse_adam_table_step(p, m, v, ls, so.LAST_STEP_PER_ROW, R, c,
                                           so.csr(ro, co[:u * c], vals_csr), t, cfg, so.DORMANCY_DECAY, None, err))
        ci, cv, _, _ = oracle.canonicalize(idx, vals, R)
        oro, oco = oracle.row_coo_to_csr(ci, R, c)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, so.status_string(int(err.item()))
        assert np.array_equal(host(ro), oro) and np.array_equal(host(co)[:u * c], oco)
        assert oracle.adam_table_step(op, om, ov, ols, t, row_off=oro, cols=oco, vals=cv.reshape(-1),
                                      mode=oracle.MODE_DORMANCY_DECAY, lr=w.lr, beta1=w.beta1, beta2=w.beta2,
                                      eps=w.eps) == 0
    assert_state_close("p", host(p), op)
    assert_state_close("m", host(m), om)
    assert_state_close("v", host(v), ov)
    assert np.array_equal(host(ls), ols)


# ------------------------------------------------------------------ 1-D
@pytest.mark.parametrize("mode", [0, 1], ids=["lazy", "dormancy_decay"])
@pytest.mark.parametrize("canonical", [True, False])
def test_adam_1d(cuda_lib, mode, canonical):
    so = cuda_lib
    import torch
    from lazy_optimizers_embedding_gb300 import workloads as wl
    w = wl.CFG_1D
    dim = w.rows
    rng = np.random.default_rng(9)
    p0 = wl.table_init(w).reshape(-1)
    p, m, v = dev(p0), torch.zeros(dim, device="cuda"), torch.zeros(dim, device="cuda")
    ls = torch.zeros(dim, dtype=torch.int64, device="cuda")
    op, om, ov, ols = p0.copy(), np.zeros_like(p0), np.zeros_like(p0), np.zeros(dim, np.int64)
    err = so.error_word()
    cfg = so.AdamConfig(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps)
    omode = oracle.MODE_DORMANCY_DECAY if mode else oracle.MODE_LAZY
    ws = so.workspace(3000, 1, dim)
    for s in range(w.steps):
        t = s + 1
        if canonical:
            idx, g = wl.coo_step(w, s)
            g = g.reshape(-1)
        else:
            idx = rng.integers(0, dim, 3000).astype(np.int64)
            idx[:500] = 17
            g = rng.standard_normal(3000).astype(np.float32)
        d_idx, d_g = dev(idx), dev(g)
        so.check(so.sparse_adam_step(p, m, v, ls, dim, d_idx, d_g, idx.shape[0], int(canonical), t, cfg, mode,
                                     None if canonical else ws, err))
        assert oracle.adam_step(op, om, ov, ols, idx, g, t, is_canonical=canonical, mode=omode, lr=w.lr,
                                beta1=w.beta1, beta2=w.beta2, eps=w.eps) == 0
        torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_state_close("p", host(p), op)
    assert_state_close("m", host(m), om)
    assert_state_close("v", host(v), ov)
    assert np.array_equal(host(ls), ols)


@pytest.mark.parametrize("n", [1, 1000, 4096, 4097])
@pytest.mark.parametrize("opt", ["adam_lazy", "adam_dd", "sgd"])
def test_canonical_1d_single_launch_boundary(cuda_lib, n, opt):
    """Canonical 1-D SGD steps of up to 4,096 entries take one single-block launch (check,
    barrier, update), 4,097 the check and row kernels; Adam steps take the two launches at every
    size.  All match the oracle, leave untouched coordinates (special values planted) bit for bit
    and stay inside their guard regions, and failed steps write nothing."""
    so = cuda_lib
    dim = 60_000
    rng = np.random.default_rng(n + len(opt))
    p0 = (rng.standard_normal(dim) * 0.01).astype(np.float32)
    steps = []
    for s in range(3):
        idx = np.sort(rng.choice(dim, n, replace=False)).astype(np.int64)
        steps.append((idx, (rng.standard_normal(n) * 0.01).astype(np.float32)))
    never = np.ones(dim, bool)
    for idx, _ in steps:
        never[idx] = False
    srng = np.random.default_rng(3)
    plant_specials(p0, never, srng)
    G = Guarded(seed=n)
    err = G.error_word()
    touched = ~never
    if opt == "sgd":
        b0 = np.zeros(dim, np.float32)
        plant_specials(b0, never, srng)
        p, buf = G.array(p0), G.array(b0)
        op, ob = p0.copy(), b0.copy()
        cfg = so.SgdConfig(lr=0.05, momentum=0.9, weight_decay=1e-4)
        for idx, g in steps:
            so.check(so.sparse_sgd_step(p, buf, dim, G.array(idx), G.array(g), n, 1, cfg, None, err))
            assert oracle.sgd_step(op, ob, idx, g, lr=0.05, momentum=0.9, weight_decay=1e-4) == 0
            G.check("sgd 1-D")
        assert int(err.item()) == 0
        assert_state_close("p", host(p), op, touched, p0)
        assert_state_close("buf", host(buf), ob, touched, b0)
        return
    mode = so.DORMANCY_DECAY if opt == "adam_dd" else so.LAZY
    omode = oracle.MODE_DORMANCY_DECAY if opt == "adam_dd" else oracle.MODE_LAZY
    m0 = np.zeros(dim, np.float32)
    v0 = np.zeros(dim, np.float32)
    plant_specials(m0, never, srng)
    plant_specials(v0, never, srng)
    p, m, v = G.array(p0), G.array(m0), G.array(v0)
    ls = G.array(np.zeros(dim, np.int64))
    op, om, ov, ols = p0.copy(), m0.copy(), v0.copy(), np.zeros(dim, np.int64)
    cfg = so.AdamConfig(**ADAM)
    for s, (idx, g) in enumerate(steps):
        t = 2 * s + 1
        so.check(so.sparse_adam_step(p, m, v, ls, dim, G.array(idx), G.array(g), n, 1, t, cfg, mode, None, err))
        assert oracle.adam_step(op, om, ov, ols, idx, g, t, mode=omode, **ADAM) == 0
        G.check("adam 1-D")
    assert int(err.item()) == 0
    assert_state_close("p", host(p), op, touched, p0)
    assert_state_close("m", host(m), om, touched, m0)
    assert_state_close("v", host(v), ov, touched, v0)
    assert np.array_equal(host(ls), ols)
    # errors on the same path: nothing written, the code set
    if n < 2:
        return
    before = [host(a).copy() for a in (p, m, v, ls)]
    idx0 = steps[0][0]
    g0 = steps[0][1]
    bad_cases = [(np.concatenate([idx0[:-1], [dim]]), so.ERR_INDEX_OUT_OF_RANGE),
                 (np.concatenate([idx0[:1], idx0[:-1]]), so.ERR_NOT_CANONICAL)]
    for bad, want in bad_cases:
        e = G.error_word()
        so.check(so.sparse_adam_step(p, m, v, ls, dim, G.array(bad.astype(np.int64)), G.array(g0), n, 1, 100, cfg,
                                     mode, None, e))
        assert int(e.item()) == want
    e = G.error_word()   # t not above the last_step of a listed coordinate
    so.check(so.sparse_adam_step(p, m, v, ls, dim, G.array(steps[-1][0]), G.array(g0), n, 1, 2 * 2 + 1, cfg, mode,
                                 None, e))
    assert int(e.item()) == so.ERR_STEP_ORDER
    G.check("adam 1-D errors")
    for name, a, b in zip(("p", "m", "v", "last_step"), (p, m, v, ls), before):
        assert host(a).tobytes() == b.tobytes(), f"{name} written by a failed step"


# ------------------------------------------------------------------ lazy SGD
@pytest.mark.parametrize("R,c,mom,wd", [(20000, 32, 0.9, 1e-4), (5000, 1, 0.9, 0.0), (3000, 128, 0.0, 0.0),
                                        (4000, 6, 0.5, 0.1)])
def test_sgd_raw_rows(cuda_lib, R, c, mom, wd):
    so = cuda_lib
    rng = np.random.default_rng(R + c)
    n = 6000
    steps = [(_raw_rows(rng, n, R, hot=R - 1, hot_count=1100 if s == 2 else 0),
              rng.standard_normal((n, c)).astype(np.float32)) for s in range(6)]
    never = np.ones(R, bool)
    for rows, _ in steps:
        never[rows] = False
    never2 = np.repeat(never[:, None], c, 1)
    p0 = (rng.standard_normal((R, c)) * 0.01).astype(np.float32)
    b0 = np.zeros_like(p0)
    srng = np.random.default_rng(5)
    plant_specials(p0, never2, srng)
    plant_specials(b0, never2, srng)
    G = Guarded(seed=R + 3 * c)
    p = G.array(p0)
    buf = G.array(b0) if mom else None
    op, ob = p0.copy(), b0.copy()
    err = G.error_word()
    cfg = so.SgdConfig(lr=0.05, momentum=mom, weight_decay=wd)
    ws = G.workspace(so, n, c, R)
    touched = np.zeros(R, bool)
    for s, (rows, vals) in enumerate(steps):
        so.check(so.sparse_sgd_table_step(p, buf, R, c, so.row_coo(G.array(rows), G.array(vals), False), cfg, ws,
                                          err))
        assert oracle.sgd_table_step(op, ob if mom else None, rows=rows, vals=vals, lr=0.05, momentum=mom,
                                     weight_decay=wd) == 0
        touched[rows] = True
        G.check(f"sgd step {s + 1}")
    assert int(err.item()) == 0
    tm = np.repeat(touched[:, None], c, 1)
    assert_state_close("p", host(p), op, tm, p0)
    if mom:
        assert_state_close("buf", host(buf), ob, tm, b0)
    else:
        assert never.any() or R <= 5000


def test_sgd_1d_canonical_and_csr(cuda_lib):
    so = cuda_lib
    import torch
    from lazy_optimizers_embedding_gb300 import workloads as wl
    w = wl.CFG_1D_SGD
    p0 = wl.table_init(w).reshape(-1)
    p, buf = dev(p0), torch.zeros(w.rows, device="cuda")
    op, ob = p0.copy(), np.zeros_like(p0)
    err = so.error_word()
    cfg = so.SgdConfig(lr=w.lr, momentum=w.momentum, weight_decay=w.weight_decay)
    for s in range(w.steps):
        idx, g = wl.coo_step(w, s)
        d_idx, d_g = dev(idx), dev(g.reshape(-1))
        so.check(so.sparse_sgd_step(p, buf, w.rows, d_idx, d_g, idx.shape[0], 1, cfg, None, err))
        assert oracle.sgd_step(op, ob, idx, g.reshape(-1), lr=w.lr, momentum=w.momentum,
                               weight_decay=w.weight_decay) == 0
        torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_state_close("p", host(p), op)
    assert_state_close("buf", host(buf), ob)
    # SparseSgdTable with an element-granular CSR gradient: the CSR kernel (no workspace) and the
    # flat one-entry-per-thread update (workspace given)
    R, c = 3000, 20
    for with_ws in (False, True):
        rng = np.random.default_rng(2)
        t0 = rng.standard_normal((R, c)).astype(np.float32)
        G = Guarded(seed=17)
        tp, tb = G.array(t0), G.zeros((R, c))
        tq, tbq = t0.copy(), np.zeros_like(t0)
        ws = G.workspace(so, 400 * 5 + 64, 1, R) if with_ws else None
        for s in range(3):
            ro, co, va = _csr_elem(rng, R, c, 400, 5)
            so.check(so.sparse_sgd_table_step(tp, tb, R, c, so.csr(G.array(ro), G.array(co), G.array(va)), cfg, ws,
                                              err))
            assert oracle.sgd_table_step(tq, tbq, row_off=ro, cols=co, vals=va, lr=w.lr, momentum=w.momentum,
                                         weight_decay=w.weight_decay) == 0
            G.check(f"sgd csr step {s + 1}")
        assert int(err.item()) == 0
        assert_state_close("p", host(tp), tq)
        assert_state_close("buf", host(tb), tbq)


# ------------------------------------------------------------------ conversions
@pytest.mark.parametrize("r,c,k", [(0, 3, 0), (1, 1, 1), (50, 7, 100), (10_000, 64, 30_000), (3000, 1, 1500),
                                   (40, 100_000, 5000)])
def test_csr_coo_round_trip_matches_oracle(cuda_lib, r, c, k):
    so = cuda_lib
    import torch
    rng = np.random.default_rng(r + c + k)
    lin = np.sort(rng.choice(r * c, size=k, replace=False)).astype(np.int64) if r else np.zeros(0, np.int64)
    oro, oco = oracle.coo_to_csr(lin, r, c)
    err = so.error_word()
    d_lin = dev(lin)
    ro = torch.empty(r + 1, dtype=torch.int64, device="cuda")
    co = torch.empty(max(k, 1), dtype=torch.int32, device="cuda")
    so.check(so.sparse_coo_to_csr(d_lin, k, r, c, ro, co, err))
    back = torch.empty(max(k, 1), dtype=torch.int64, device="cuda")
    so.check(so.sparse_csr_to_coo(ro, co, r, c, k, back, err))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(host(ro), oro)
    assert np.array_equal(host(co)[:k], oco)
    assert np.array_equal(host(back)[:k], lin)


def test_golden_csr_coo_on_gpu(cuda_lib):
    """The hand-derived CSR <-> COO fixture ("Sparse gradient representations") on the GPU."""
    so = cuda_lib
    import torch
    from conftest import read_cases
    for case in read_cases("csr_coo_linear_index.txt"):
        r, c = map(int, case["shape"][0])
        row_off = np.array(case["row_offsets"][0], np.int64)
        cols = np.array(case["col_indices"][0], np.int32)
        lin = np.array(case["linear"][0], np.int64)
        err = so.error_word()
        d_ro, d_co, d_lin = dev(row_off), dev(cols), dev(lin)
        out = torch.empty(lin.shape[0], dtype=torch.int64, device="cuda")
        so.check(so.sparse_csr_to_coo(d_ro, d_co, r, c, lin.shape[0], out, err))
        ro = torch.empty(r + 1, dtype=torch.int64, device="cuda")
        co = torch.empty(lin.shape[0], dtype=torch.int32, device="cuda")
        so.check(so.sparse_coo_to_csr(d_lin, lin.shape[0], r, c, ro, co, err))
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert np.array_equal(host(out), lin)
        assert np.array_equal(host(ro), row_off) and np.array_equal(host(co), cols)


def test_golden_duplicate_sum_on_gpu(cuda_lib):
    so = cuda_lib
    import torch
    from conftest import read_cases
    for case in read_cases("duplicate_sum.txt"):
        bound = int(case["bound"][0][0])
        c = int(case["cols"][0][0])
        idx = np.array(case["idx"][0], np.int64)
        n = idx.shape[0]
        vals = np.array([float(x) for x in case["vals"][0]], np.float32).reshape(n, c)
        d_idx, d_vals = dev(idx), dev(vals)
        io = torch.empty(n, dtype=torch.int64, device="cuda")
        vo = torch.empty((n, c), device="cuda")
        so_ = torch.empty(n + 1, dtype=torch.int64, device="cuda")
        po = torch.empty(n, dtype=torch.int64, device="cuda")
        nnz = torch.zeros(1, dtype=torch.int64, device="cuda")
        err = so.error_word()
        so.check(so.sparse_canonicalize(d_idx, d_vals, n, c, bound, io, vo, so_, po, nnz,
                                        so.workspace(n, c, bound), err))
        torch.cuda.synchronize()
        u = int(nnz.item())
        assert list(host(io)[:u]) == [int(x) for x in case["canonical_idx"][0]]
        want = np.array([float(x) for x in case["canonical_vals"][0]], np.float32).reshape(-1, c)
        assert host(vo)[:u].tobytes() == want.tobytes()
        assert list(host(so_)[:u + 1]) == [int(x) for x in case["seg_off"][0]]
        assert list(host(po)) == [int(x) for x in case["perm"][0]]


# ------------------------------------------------------------------ errors: all or nothing
def test_errors_set_d_err_and_write_nothing(cuda_lib):
    so = cuda_lib
    import torch
    R, c = 100, 8
    rng = np.random.default_rng(4)
    p0 = rng.standard_normal((R, c)).astype(np.float32)
    p, m, v = dev(p0), torch.zeros((R, c), device="cuda"), torch.zeros((R, c), device="cuda")
    ls0 = np.zeros(R, np.int64)
    ls0[40] = 9
    ls = dev(ls0)
    cfg = so.AdamConfig(**ADAM)
    ws = so.workspace(64, c, R)
    g2 = dev(np.ones((2, c), np.float32))

    def step(grad, t=5, layout=so.LAST_STEP_PER_ROW, lsv=ls):
        err = so.error_word()
        so.check(so.sparse_adam_table_step(p, m, v, lsv, layout, R, c, grad, t, cfg, so.DORMANCY_DECAY, ws, err))
        torch.cuda.synchronize()
        return int(err.item())

    cases = [
        (so.row_coo(dev(np.array([3, R])), g2, False), so.ERR_INDEX_OUT_OF_RANGE),
        (so.row_coo(dev(np.array([-1, 3])), g2, False), so.ERR_INDEX_OUT_OF_RANGE),
        (so.row_coo(dev(np.array([3, R + 5])), g2, True), so.ERR_INDEX_OUT_OF_RANGE),
        (so.row_coo(dev(np.array([7, 7])), g2, True), so.ERR_NOT_CANONICAL),
        (so.row_coo(dev(np.array([9, 2])), g2, True), so.ERR_NOT_CANONICAL),
        (so.row_coo(dev(np.array([40, 2])), g2, False), so.ERR_STEP_ORDER),
        (so.row_coo(dev(np.array([2, 40])), g2, True), so.ERR_STEP_ORDER),
    ]
    for grad, want in cases:
        assert step(grad) == want

    # CSR: partial row under per-row last_step; unordered columns; column out of range; bad offsets
    def csr_case(row_off, cols):
        return so.csr(dev(np.array(row_off, np.int64)), dev(np.array(cols, np.int32)),
                      dev(np.ones(len(cols), np.float32)))

    partial = [0] * (R + 1)
    for i in range(1, R + 1):
        partial[i] = 1 if i > 3 else 0
    assert step(csr_case(partial, [2])) == so.ERR_NOT_CANONICAL
    # full rows (per-row last_step): row 3 holds all c columns
    full = [0 if i <= 3 else c for i in range(R + 1)]
    assert step(csr_case(full, list(range(c - 1)) + [c])) == so.ERR_INDEX_OUT_OF_RANGE
    assert step(csr_case(full, [1, 0] + list(range(2, c)))) == so.ERR_NOT_CANONICAL
    at40 = [0 if i <= 40 else c for i in range(R + 1)]      # row 40: last_step 9 >= t
    assert step(csr_case(at40, list(range(c)))) == so.ERR_STEP_ORDER
    shifted = [1 if i <= 3 else c + 1 for i in range(R + 1)]  # offsets not starting at 0
    assert step(csr_case(shifted, [0] + list(range(c)))) == so.ERR_NOT_CANONICAL   # columns all in range
    lsc = dev(np.zeros(R * c, np.int64))
    unordered = [0, 0, 0, 0] + [2] * (R - 3)
    assert step(csr_case(unordered, [5, 1]), layout=so.LAST_STEP_PER_COORD, lsv=lsc) == so.ERR_NOT_CANONICAL
    assert step(csr_case(partial, [c]), layout=so.LAST_STEP_PER_COORD, lsv=lsc) == so.ERR_INDEX_OUT_OF_RANGE
    bad_end = list(partial)
    bad_end[-1] = 5
    assert step(csr_case(bad_end, [1]), layout=so.LAST_STEP_PER_COORD, lsv=lsc) == so.ERR_NOT_CANONICAL
    assert np.array_equal(host(p), p0) and not host(m).any() and not host(v).any()
    assert np.array_equal(host(ls), ls0) and not host(lsc).any()
    # sticky: a valid step with a set error word writes nothing
    err = so.error_word()
    err.fill_(so.ERR_NOT_CANONICAL)
    so.check(so.sparse_adam_table_step(p, m, v, ls, so.LAST_STEP_PER_ROW, R, c,
                                       so.row_coo(dev(np.array([1, 2])), g2, True), 11, cfg, so.LAZY, None, err))
    torch.cuda.synchronize()
    assert int(err.item()) == so.ERR_NOT_CANONICAL and np.array_equal(host(p), p0)
    # host-side rejections return before launching
    e = so.error_word()
    bad = so.AdamConfig(lr=1e-3, beta1=1.0, beta2=0.999, eps=1e-8)
    g = so.row_coo(dev(np.array([1])), dev(np.ones((1, c), np.float32)), True)
    assert so.sparse_adam_table_step(p, m, v, ls, 0, R, c, g, 12, bad, 1, None, e) == so.ERR_INVALID_ARG
    assert so.sparse_adam_table_step(p, m, v, ls, 0, R, c, g, 0, cfg, 1, None, e) == so.ERR_INVALID_ARG
    graw = so.row_coo(dev(np.array([1])), dev(np.ones((1, c), np.float32)), False)
    assert so.sparse_adam_table_step(p, m, v, ls, 0, R, c, graw, 12, cfg, 1, None, e) == so.ERR_WORKSPACE


def test_determinism_raw_zipf(cuda_lib):
    """Every addition has a fixed order: two runs give bitwise equal state."""
    so = cuda_lib
    import torch
    from lazy_optimizers_embedding_gb300 import workloads as wl
    w = wl.CFG_ZIPF_10M_128.scaled(rows=50_000, lookups=40_000)
    p0 = wl.table_init(w)
    res = []
    for _ in range(2):
        p = dev(p0)
        m, v = torch.zeros_like(p), torch.zeros_like(p)
        ls = torch.zeros(w.rows, dtype=torch.int64, device="cuda")
        err = so.error_word()
        ws = so.workspace(w.lookups, w.cols, w.rows)
        for s in range(3):
            idx, vals = wl.coo_step(w, s)
            so.check(so.sparse_adam_table_step(p, m, v, ls, 0, w.rows, w.cols, so.row_coo(dev(idx), dev(vals), False),
                                               s + 1, so.AdamConfig(**ADAM), so.DORMANCY_DECAY, ws, err))
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        res.append((host(p), host(m), host(v)))
    for a, b in zip(*res):
        assert a.tobytes() == b.tobytes()


@pytest.mark.parametrize("beta1,gap_steps", [(0.0, 1), (0.9, 1), (0.9, 500), (0.5, 3000)])
def test_edge_betas_and_long_gaps(cuda_lib, beta1, gap_steps):
    """beta1 = 0; gap 1 (DormancyDecay == Lazy); long dormancy (beta^gap underflows)."""
    so = cuda_lib
    import torch
    R, c = 64, 4
    hp = dict(lr=1e-2, beta1=beta1, beta2=0.99, eps=1e-8)
    rng = np.random.default_rng(11)
    p0 = rng.standard_normal((R, c)).astype(np.float32)
    grads = [rng.standard_normal((2, c)).astype(np.float32) for _ in range(3)]
    outs = {}
    for mode in (so.LAZY, so.DORMANCY_DECAY):
        p, m, v = dev(p0), torch.zeros((R, c), device="cuda"), torch.zeros((R, c), device="cuda")
        ls = torch.zeros(R, dtype=torch.int64, device="cuda")
        op, om, ov, ols = p0.copy(), np.zeros_like(p0), np.zeros_like(p0), np.zeros(R, np.int64)
        err = so.error_word()
        for k, t in enumerate((1, 1 + gap_steps, 2 + gap_steps)):
            rows = np.array([0, R - 1], np.int64)
            g = grads[k]
            so.check(so.sparse_adam_table_step(p, m, v, ls, 0, R, c, so.row_coo(dev(rows), dev(g), True), t,
                                               so.AdamConfig(**hp), mode, None, err))
            assert oracle.adam_table_step(op, om, ov, ols, t, rows=rows, vals=g, is_canonical=True,
                                          mode=oracle.MODE_DORMANCY_DECAY if mode else oracle.MODE_LAZY, **hp) == 0
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_state_close("p", host(p), op)
        assert_state_close("m", host(m), om)
        assert_state_close("v", host(v), ov)
        outs[mode] = host(p)
    if gap_steps == 1:  # every touch has gap 1: the two modes coincide bit for bit
        assert outs[so.LAZY].tobytes() == outs[so.DORMANCY_DECAY].tobytes()


# ------------------------------------------------------------------ row gather (read_rows)
@pytest.mark.parametrize("r,c,n", [(1, 1, 1), (50, 3, 500), (1000, 4, 4097), (3000, 64, 10_000), (2000, 128, 7001),
                                   (400, 300, 999), (100, 1000, 257)])
def test_read_rows_bitwise(cuda_lib, r, c, n):
    import torch
    so = cuda_lib
    rng = np.random.default_rng(r * 7 + c)
    t = rng.standard_normal((r, c)).astype(np.float32)
    t.view(np.uint32)[0, 0] = 0x7FC0BEEF        # NaN payload
    if c > 2:
        t[r - 1, 1], t[r - 1, 2] = np.float32(-0.0), np.float32(3e-41)
    idx = rng.integers(0, r, n).astype(np.int64)
    idx[: min(n, 3)] = [0, r - 1, 0][: min(n, 3)]
    out = torch.full((n, c), 7.0, device="cuda")
    err = so.error_word()
    so.check(so.sparse_read_rows(dev(t), r, c, dev(idx), n, out, err), "read_rows")
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert host(out).tobytes() == oracle.read_rows(t, idx).tobytes()


def test_read_rows_bad_index_and_empty(cuda_lib):
    import torch
    so = cuda_lib
    t = np.arange(40, dtype=np.float32).reshape(10, 4)
    idx = np.array([2, 10, 5, -1, 9], np.int64)
    out = torch.full((5, 4), -3.0, device="cuda")
    err = so.error_word()
    so.check(so.sparse_read_rows(dev(t), 10, 4, dev(idx), 5, out, err), "read_rows")
    torch.cuda.synchronize()
    assert int(err.item()) == so.ERR_INDEX_OUT_OF_RANGE
    got = host(out)
    assert np.array_equal(got[[0, 2, 4]], t[[2, 5, 9]])
    assert np.all(got[[1, 3]] == -3.0)
    err2 = so.error_word()
    assert so.sparse_read_rows(dev(t), 10, 4, dev(idx), 0, out, err2) == so.OK
    assert so.sparse_read_rows(dev(t), 10, 0, dev(idx), 5, out, err2) == so.ERR_INVALID_ARG


# ------------------------------------------------------------------ non-finite gradient check
@pytest.mark.parametrize("n,offset", [(1, 0), (7, 1), (1000, 0), (4099, 3), (262_147, 2)])
def test_check_finite_matches_oracle(cuda_lib, n, offset):
    """Values are read from an offset into a buffer, so the head / body / tail split is exercised."""
    import torch
    so = cuda_lib
    rng = np.random.default_rng(n + offset)
    base = rng.standard_normal(n + offset).astype(np.float32)
    base[offset] = np.float32(3.0e38)
    d = dev(base)
    view = d[offset:]
    for pos, bad in [(None, None), (0, np.nan), (n - 1, np.inf), (n // 2, -np.inf)]:
        h = base[offset:].copy()
        if pos is not None:
            h[pos] = bad
        view.copy_(torch.from_numpy(h))
        err = so.error_word()
        so.check(so.sparse_check_finite(view, n, err), "check_finite")
        torch.cuda.synchronize()
        assert int(err.item()) == oracle.check_finite(h)


def test_check_finite_then_step_writes_nothing(cuda_lib):
    """A non-finite value found before the step leaves every state array untouched (sticky error word)."""
    import torch
    so = cuda_lib
    rng = np.random.default_rng(77)
    R, c, n = 500, 32, 2000
    p0 = rng.standard_normal((R, c)).astype(np.float32)
    rows = rng.integers(0, R, n)
    vals = rng.standard_normal((n, c)).astype(np.float32)
    vals[1234, 5] = np.nan
    p, m, v = dev(p0), torch.zeros((R, c), device="cuda"), torch.zeros((R, c), device="cuda")
    ls = torch.zeros(R, dtype=torch.int64, device="cuda")
    dvals = dev(vals)
    err = so.error_word()
    so.check(so.sparse_check_finite(dvals, n * c, err), "check_finite")
    g = so.row_coo(dev(rows), dvals, False)
    so.check(so.sparse_adam_table_step(p, m, v, ls, so.LAST_STEP_PER_ROW, R, c, g, 1,
                                       so.AdamConfig(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8), so.DORMANCY_DECAY,
                                       so.workspace(n, c, R), err), "step")
    torch.cuda.synchronize()
    assert int(err.item()) == so.ERR_NON_FINITE
    assert host(p).tobytes() == p0.tobytes()
    assert not host(m).any() and not host(v).any() and not host(ls).any()


# ------------------------------------------------------------------ moment-state check
def _state_case(rng, R, c, form):
    m = (rng.standard_normal((R, c)) * 0.1).astype(np.float32)
    v = (np.abs(rng.standard_normal((R, c))) * 1e-4).astype(np.float32)
    if form == "csr":
        nrows = max(1, R // 3)
        rows = np.sort(rng.choice(R, nrows, replace=False))
        k = max(1, c // 3)
        counts = np.zeros(R, np.int64)
        counts[rows] = k
        row_off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
        cols = np.sort(np.argsort(rng.random((nrows, c)), axis=1)[:, :k], axis=1).astype(np.int32).reshape(-1)
        return m, v, dict(row_off=row_off, cols=cols)
    rows = rng.integers(0, R, 3 * R).astype(np.int64)
    rows = rows[rows % 5 != 0]          # rows 0, 5, 10, ... are never listed
    if form == "canon":
        rows = np.unique(rows)
    return m, v, dict(rows=rows)


@pytest.mark.parametrize("form", ["raw", "canon", "csr"])
@pytest.mark.parametrize("R,c", [(1, 1), (100, 1), (300, 4), (500, 64), (200, 128), (90, 300), (64, 7)])
def test_check_state_matches_oracle(cuda_lib, form, R, c):
    """sparse_check_state against the oracle, with specials planted inside and outside the read set."""
    import torch
    so = cuda_lib
    rng = np.random.default_rng(R * 13 + c + len(form))
    m, v, g = _state_case(rng, R, c, form)
    if "rows" in g:
        read = np.zeros((R, c), bool)
        read[g["rows"]] = True
    else:
        read = np.zeros((R, c), bool)
        read[np.repeat(np.arange(R), np.diff(g["row_off"])), g["cols"]] = True
    cases = [("clean", None, None)]
    for bits, arr in ((0x7FC00001, "m"), (0x7F800000, "m"), (0xFF800000, "v"), (0x7FC12345, "v"),
                      (0xBF800000, "v"), (0x80000001, "v"), (0x80000000, "v")):
        cases.append(("inside", bits, arr))
        cases.append(("outside", bits, arr))
    for where, bits, arr in cases:
        mm, vv = m.copy(), v.copy()
        if bits is not None:
            pool = np.flatnonzero(read.reshape(-1) if where == "inside" else ~read.reshape(-1))
            if pool.size == 0:
                continue
            (mm if arr == "m" else vv).reshape(-1).view(np.uint32)[rng.choice(pool)] = bits
        want = oracle.check_state(mm, vv, **g)
        G = Guarded(seed=R + c)
        dm, dv = G.array(mm), G.array(vv)
        if "rows" in g:
            grad = so.row_coo(G.array(g["rows"]), G.empty((g["rows"].shape[0], c), torch.float32), form == "canon")
        else:
            grad = so.csr(G.array(g["row_off"]), G.array(g["cols"]), G.empty(g["cols"].shape[0], torch.float32))
        err = G.error_word()
        so.check(so.sparse_check_state(dm, dv, R, c, grad, err), "check_state")
        G.check("check_state")
        assert int(err.item()) == want, (where, hex(bits or 0), arr)
        assert host(dm).tobytes() == mm.tobytes() and host(dv).tobytes() == vv.tobytes()


def test_check_state_bad_index_and_empty(cuda_lib):
    import torch
    so = cuda_lib
    m = torch.zeros((10, 4), device="cuda")
    v = torch.zeros((10, 4), device="cuda")
    for rows, want in (([2, 10], so.ERR_INDEX_OUT_OF_RANGE), ([-1], so.ERR_INDEX_OUT_OF_RANGE), ([], so.OK)):
        r = np.array(rows, np.int64)
        err = so.error_word()
        grad = so.row_coo(dev(r) if r.size else torch.zeros(1, dtype=torch.int64, device="cuda"),
                          torch.zeros((max(r.size, 1), 4), device="cuda"), False)
        grad.n = r.size
        so.check(so.sparse_check_state(m, v, 10, 4, grad, err))
        torch.cuda.synchronize()
        assert int(err.item()) == want
    # a malformed CSR is reported by the structure check; the state pass reads nothing
    err = so.error_word()
    bad = so.csr(dev(np.array([0] * 10 + [5], np.int64)), dev(np.array([0, 1], np.int32)), torch.zeros(2, device="cuda"))
    so.check(so.sparse_check_state(m, v, 10, 4, bad, err))
    torch.cuda.synchronize()
    assert int(err.item()) == so.ERR_NOT_CANONICAL


@pytest.mark.parametrize("form", ["raw", "csr"])
def test_check_state_then_step_writes_nothing(cuda_lib, form):
    """A corrupted touched moment found before the step leaves every state array untouched."""
    import torch
    so = cuda_lib
    rng = np.random.default_rng(78)
    R, c = 400, 32
    p0 = rng.standard_normal((R, c)).astype(np.float32)
    m0 = (rng.standard_normal((R, c)) * 1e-3).astype(np.float32)
    v0 = (np.abs(rng.standard_normal((R, c))) * 1e-6).astype(np.float32)
    if form == "raw":
        rows = rng.integers(0, R, 1500)
        v0[rows[700], 3] = np.float32(-1e-9)
        grad_np = dict(rows=rows)
        vals = dev(rng.standard_normal((rows.shape[0], c)).astype(np.float32))
        grad = so.row_coo(dev(rows), vals, False)
        layout, ls_n, ws = so.LAST_STEP_PER_ROW, R, so.workspace(rows.shape[0], c, R)
    else:
        _, _, grad_np = _state_case(rng, R, c, "csr")
        first = int(np.flatnonzero(np.diff(grad_np["row_off"]))[0])
        m0[first, grad_np["cols"][grad_np["row_off"][first]]] = np.float32(np.nan)
        grad = so.csr(dev(grad_np["row_off"]), dev(grad_np["cols"]),
                      dev(rng.standard_normal(grad_np["cols"].shape[0]).astype(np.float32)))
        layout, ls_n, ws = so.LAST_STEP_PER_COORD, R * c, None
    assert oracle.check_state(m0, v0, **grad_np) == oracle.ERR_BAD_STATE
    p, m, v = dev(p0), dev(m0), dev(v0)
    ls = torch.zeros(ls_n, dtype=torch.int64, device="cuda")
    err = so.error_word()
    so.check(so.sparse_check_state(m, v, R, c, grad, err), "check_state")
    so.check(so.sparse_adam_table_step(p, m, v, ls, layout, R, c, grad, 1,
                                       so.AdamConfig(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8), so.DORMANCY_DECAY,
                                       ws, err), "step")
    torch.cuda.synchronize()
    assert int(err.item()) == so.ERR_BAD_STATE
    assert host(p).tobytes() == p0.tobytes() and host(m).tobytes() == m0.tobytes()
    assert host(v).tobytes() == v0.tobytes() and not host(ls).any()


# ------------------------------------------------------------------ chained calls, no host sync
def test_chained_outputs_without_host_sync(cuda_lib):
    """Library outputs fed straight into the next call on the same stream, no synchronisation:
    CSR -> COO -> canonicalize(lin), and canonicalize(values not requested) -> raw step on its
    unique indices.  The second call's first kernel reads its index array before waiting for the
    previous kernel, so every producer must finish its writes before releasing its dependents."""
    import torch
    so = cuda_lib
    rng = np.random.default_rng(123)
    iters = 40
    r, c = 3000, 64
    cases = []
    for it in range(iters):
        k = int(rng.integers(1, 60_000))
        lin = np.sort(rng.choice(r * c, size=k, replace=False)).astype(np.int64)
        ro, co = oracle.coo_to_csr(lin, r, c)
        cases.append((lin, ro, co))
    err = so.error_word()
    bufs = []
    for lin, ro, co in cases:   # every input and output allocated first
        k = lin.shape[0]
        bufs.append((k, dev(ro), dev(co), torch.empty(k, dtype=torch.int64, device="cuda"),
                     [torch.empty(k, dtype=torch.int64, device="cuda") for _ in range(4)],
                     torch.zeros(1, dtype=torch.int64, device="cuda"), so.workspace(k, 1, r * c)))
    torch.cuda.synchronize()   # from here on nothing waits on the host
    outs = []
    for k, d_ro, d_co, lin_out, chain, nnz, ws in bufs:
        so.check(so.sparse_csr_to_coo(d_ro, d_co, r, c, k, lin_out, err))
        src = lin_out
        for dst in chain:      # each canonical output is the next call's raw input
            so.check(so.sparse_canonicalize(src, None, k, 1, r * c, dst, None, None, None, nnz, ws, err))
            src = dst
        outs.append((lin_out, src, nnz))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for (lin, _, _), (lin_out, idx_out, nnz) in zip(cases, outs):
        assert np.array_equal(host(lin_out), lin)
        assert int(nnz.item()) == lin.shape[0]
        assert np.array_equal(host(idx_out), lin)

    # canonicalize without values -> lazy Adam on the unique rows, raw form
    R, cc, n = 20_000, 32, 30_000
    cfg = so.AdamConfig(**ADAM)
    p0 = (rng.standard_normal((R, cc)) * 0.01).astype(np.float32)
    p, m, v = dev(p0), torch.zeros((R, cc), device="cuda"), torch.zeros((R, cc), device="cuda")
    ls = torch.zeros(R, dtype=torch.int64, device="cuda")
    op, om, ov, ols = p0.copy(), np.zeros_like(p0), np.zeros_like(p0), np.zeros(R, np.int64)
    steps = []
    for s in range(12):
        idx = _raw_rows(rng, n, R, hot=s, hot_count=2000)
        u = np.unique(idx)
        vals = (rng.standard_normal((u.shape[0], cc)) * 0.01).astype(np.float32)
        steps.append((idx, u, vals))
    dev_in = [(dev(idx), dev(vals), torch.empty(n, dtype=torch.int64, device="cuda")) for idx, _, vals in steps]
    wsc, wss = so.workspace(n, 1, R), so.workspace(n, cc, R)
    nnz = torch.zeros(1, dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    for t, ((idx, u, vals), (d_idx, d_vals, idx_out)) in enumerate(zip(steps, dev_in), start=1):
        so.check(so.sparse_canonicalize(d_idx, None, n, 1, R, idx_out, None, None, None, nnz, wsc, err))
        so.check(so.sparse_adam_table_step(p, m, v, ls, so.LAST_STEP_PER_ROW, R, cc,
                                           so.row_coo(idx_out[:u.shape[0]], d_vals, False), t, cfg,
                                           so.DORMANCY_DECAY, wss, err))
        assert u.shape[0] <= n
    for t, (idx, u, vals) in enumerate(steps, start=1):
        assert oracle.adam_table_step(op, om, ov, ols, t, rows=u, vals=vals, mode=oracle.MODE_DORMANCY_DECAY,
                                      **ADAM) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0, so.status_string(int(err.item()))
    for (idx, u, _), (_, _, idx_out) in zip(steps, dev_in):
        assert np.array_equal(host(idx_out)[:u.shape[0]], u)
    assert_state_close("p", host(p), op)
    assert_state_close("m", host(m), om)
    assert_state_close("v", host(v), ov)
    assert np.array_equal(host(ls), ols)
