"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU).

Each test names the passage it follows.  Page titles:
  [optirs]  "Module sparse_optimizer" (optirs-gpu 0.3.2 docs)
  [DSA]     "DiskSparseAdam (DSA)" README
"""
import math

import numpy as np
import pytest

import oracle
from oracle import dense_emulator as de
from conftest import read_cases

DD = oracle.MODE_DORMANCY_DECAY
LAZY = oracle.MODE_LAZY


def _fl(xs):
    return [float(x) for x in xs]


# --------------------------------------------------------------------------
# golden fixtures (hand-derived worked examples)
# --------------------------------------------------------------------------
def test_golden_csr_coo_linear_index():
    """[optirs] Sparse gradient representations: lin = row*c + col, lossless both ways."""
    for case in read_cases("csr_coo_linear_index.txt"):
        r, c = map(int, case["shape"][0])
        row_off = np.array(case["row_offsets"][0], np.int64)
        cols = np.array(case["col_indices"][0], np.int32)
        lin = np.array(case["linear"][0], np.int64)
        assert np.array_equal(oracle.csr_to_coo(row_off, cols, r, c), lin)
        ro2, co2 = oracle.coo_to_csr(lin, r, c)
        assert np.array_equal(ro2, row_off) and np.array_equal(co2, cols)


def test_golden_duplicate_sum():
    """[DSA] duplicates summed, sorted after dedup; [optirs] strictly ascending canonical form."""
    for case in read_cases("duplicate_sum.txt"):
        bound = int(case["bound"][0][0])
        c = int(case["cols"][0][0])
        idx = np.array(case["idx"][0], np.int64)
        vals = np.array(_fl(case["vals"][0]), np.float32).reshape(len(idx), c)
        ci, cv, seg, perm = oracle.canonicalize(idx, vals, bound)
        assert np.array_equal(ci, np.array(case["canonical_idx"][0], np.int64))
        want = np.array(_fl(case["canonical_vals"][0]), np.float32).reshape(-1, c)
        assert cv.tobytes() == want.tobytes()
        assert np.array_equal(seg, np.array(case["seg_off"][0], np.int64))
        assert np.array_equal(perm, np.array(case["perm"][0], np.int64))


def _worked_adam(mode_name, state_dtype):
    case = read_cases("lazy_adam_worked_example.txt")[0]
    hp = dict(lr=float(case["lr"][0][0]), beta1=float(case["beta1"][0][0]),
              beta2=float(case["beta2"][0][0]), eps=float(case["eps"][0][0]))
    p = np.array(_fl(case["p_init"][0]), state_dtype)
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    ls = np.zeros(p.shape[0], np.int64)
    mode = DD if mode_name == "dormancy_decay" else LAZY
    snaps = {}
    for t_str, i_str, g_str in case["touch"]:
        t = int(t_str)
        rc = oracle.adam_step(p, m, v, ls, np.array([int(i_str)]), np.array([float(g_str)], np.float32),
                              t, mode=mode, **hp)
        assert rc == 0
        snaps[t] = (p.copy(), m.copy(), v.copy())
    return case, snaps, ls


@pytest.mark.parametrize("mode_name", ["dormancy_decay", "lazy"])
def test_golden_lazy_adam_worked_example(mode_name):
    """[optirs] Lazy Adam, both LazyAdamMode variants, against the hand-worked example."""
    case, snaps, ls = _worked_adam(mode_name, np.float64)
    exp = {}
    for line_key in ("after_t1", "after_t2"):
        for what, *vals in case[line_key]:
            exp[(int(line_key[-1]), what)] = np.array(_fl(vals))
    for row in case[mode_name]:  # lines "<mode> after_t3 <what> values..."
        assert row[0] == "after_t3"
        exp[(3, row[1])] = np.array(_fl(row[2:]))
    for (t, what), want in exp.items():
        got = snaps[t][{"p": 0, "m": 1, "v": 2}[what]]
        assert np.allclose(got, want, rtol=1e-15, atol=0), (t, what, got, want)
    assert list(ls) == [int(x) for x in case["last_step"][0]]
    # fp32 state: the moments are dyadic and exact in fp32 as well
    _, snaps32, _ = _worked_adam(mode_name, np.float32)
    for (t, what), want in exp.items():
        got = snaps32[t][{"p": 0, "m": 1, "v": 2}[what]]
        if what in ("m", "v"):
            assert np.array_equal(got, want.astype(np.float32))
        else:
            assert np.allclose(got, want, rtol=1e-7, atol=0)


def test_golden_sgd_worked_example():
    """[optirs] Sparse SGD: coupled weight decay, lazy momentum; untouched bit-identical."""
    case = read_cases("sgd_worked_example.txt")[0]
    hp = dict(lr=float(case["lr"][0][0]), momentum=float(case["momentum"][0][0]),
              weight_decay=float(case["weight_decay"][0][0]))
    for dt in (np.float32, np.float64):
        p = np.array(_fl(case["p_init"][0]), dt)
        buf = np.zeros_like(p)
        by_t = {}
        for t_str, i_str, g_str in case["touch"]:
            by_t.setdefault(int(t_str), []).append((int(i_str), float(g_str)))
        for t in sorted(by_t):
            idx = np.array([i for i, _ in by_t[t]], np.int64)
            g = np.array([x for _, x in by_t[t]], np.float32)
            assert oracle.sgd_step(p, buf, idx, g, **hp) == 0
        for what, *vals in case["after"]:
            got = p if what == "p" else buf
            assert np.array_equal(got, np.array(_fl(vals), dt)), (what, got)


# --------------------------------------------------------------------------
# P1: gap == 1 every step reduces to dense Adam (torch.optim.Adam as the library routine)
# --------------------------------------------------------------------------
def test_p1_dense_adam_reduction_vs_torch():
    """[optirs] DormancyDecay: for a coordinate touched every step gap == 1 and the update
    reduces exactly to the standard Adam recursion."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    r, c, T = 5, 3, 25
    hp = dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8)
    p0 = rng.standard_normal((r, c))
    grads = rng.standard_normal((T, r, c)).astype(np.float32)
    res = {}
    for mode in (LAZY, DD):
        p = p0.copy()
        m = np.zeros_like(p)
        v = np.zeros_like(p)
        ls = np.zeros(r, np.int64)
        for t in range(1, T + 1):
            assert oracle.adam_table_step(p, m, v, ls, t, rows=np.arange(r), vals=grads[t - 1],
                                          is_canonical=True, mode=mode, **hp) == 0
        res[mode] = (p, m, v)
    # Lazy and DormancyDecay are bit-identical when gap == 1
    for a, b in zip(res[LAZY], res[DD]):
        assert a.tobytes() == b.tobytes()
    tp = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.Adam([tp], lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"],
                           foreach=False)
    for t in range(T):
        tp.grad = torch.tensor(grads[t].astype(np.float64))
        opt.step()
    st = opt.state[tp]
    np.testing.assert_allclose(res[DD][0], tp.detach().numpy(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(res[DD][1], st["exp_avg"].numpy(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(res[DD][2], st["exp_avg_sq"].numpy(), rtol=1e-12, atol=1e-15)


# --------------------------------------------------------------------------
# P10: weight decay (DSA README, "Explicit Weight Decay Semantics", k = 0)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("wd_mode", [oracle.WD_L2, oracle.WD_DECOUPLED], ids=["l2", "decoupled"])
def test_p10_weight_decay_vs_torch(wd_mode):
    """With every coordinate touched every step, "l2" is classic Adam with L2
    (torch.optim.Adam weight_decay) and "decoupled" is AdamW (torch.optim.AdamW),
    in both lazy modes."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(12)
    r, c, T, wd = 4, 3, 20, 0.05
    hp = dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8)
    p0 = rng.standard_normal((r, c))
    grads = rng.standard_normal((T, r, c)).astype(np.float32)
    out = {}
    for mode in (LAZY, DD):
        p, m, v = p0.copy(), np.zeros((r, c)), np.zeros((r, c))
        ls = np.zeros(r, np.int64)
        for t in range(1, T + 1):
            assert oracle.adam_table_step(p, m, v, ls, t, rows=np.arange(r), vals=grads[t - 1], is_canonical=True,
                                          mode=mode, weight_decay=wd, wd_mode=wd_mode, **hp) == 0
        out[mode] = p
    assert out[LAZY].tobytes() == out[DD].tobytes()
    tp = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    cls = torch.optim.Adam if wd_mode == oracle.WD_L2 else torch.optim.AdamW
    opt = cls([tp], lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"], weight_decay=wd, foreach=False)
    for t in range(T):
        tp.grad = torch.tensor(grads[t].astype(np.float64))
        opt.step()
    np.testing.assert_allclose(out[DD], tp.detach().numpy(), rtol=1e-12, atol=1e-15)
    # the two modes really differ
    if wd_mode == oracle.WD_DECOUPLED:
        other = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
        o2 = torch.optim.Adam([other], lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"],
                              weight_decay=wd, foreach=False)
        for t in range(T):
            other.grad = torch.tensor(grads[t].astype(np.float64))
            o2.step()
        assert np.abs(out[DD] - other.detach().numpy()).max() > 1e-6


@pytest.mark.parametrize("wd_mode", [oracle.WD_L2, oracle.WD_DECOUPLED], ids=["l2", "decoupled"])
def test_p10_weight_decay_touches_only_listed_coordinates(wd_mode):
    """Decay is lazy: a row left out of a step keeps its bytes, whatever wd."""
    rng = np.random.default_rng(13)
    r, c = 6, 2
    p = rng.standard_normal((r, c)).astype(np.float32)
    p[5] = [np.float32(-0.0), np.float32(1e-40)]
    m, v = np.zeros_like(p), np.zeros_like(p)
    ls = np.zeros(r, np.int64)
    before = p.copy()
    for t in range(1, 6):
        rows = np.array([0, 2, 3], np.int64)
        g = rng.standard_normal((3, c)).astype(np.float32)
        assert oracle.adam_table_step(p, m, v, ls, t, rows=rows, vals=g, is_canonical=True, mode=DD, lr=1e-2,
                                      beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.3, wd_mode=wd_mode) == 0
    for i in (1, 4, 5):
        assert p[i].tobytes() == before[i].tobytes()
    assert not np.array_equal(p[0], before[0])


def test_p10_weight_decay_rejects_bad_settings():
    p = np.zeros((2, 1), np.float32)
    m, v = np.zeros_like(p), np.zeros_like(p)
    ls = np.zeros(2, np.int64)
    kw = dict(rows=np.array([0]), vals=np.ones((1, 1), np.float32), is_canonical=True, mode=DD, lr=1e-2,
              beta1=0.9, beta2=0.999, eps=1e-8)
    assert oracle.adam_table_step(p, m, v, ls, 1, weight_decay=-1.0, **kw) == oracle.ERR_INVALID_ARG
    assert oracle.adam_table_step(p, m, v, ls, 1, weight_decay=0.1, wd_mode=7, **kw) == oracle.ERR_INVALID_ARG


# --------------------------------------------------------------------------
# P2 / P7: dormancy equivalence and brute force against the dense emulator
# --------------------------------------------------------------------------
def _random_touches(rng, n, T, density):
    touches = []
    for _ in range(T):
        k = rng.binomial(n, density)
        sel = np.sort(rng.choice(n, size=k, replace=False))
        touches.append({int(i): float(np.float32(rng.standard_normal())) for i in sel})
    return touches


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("mode_name", ["dormancy_decay", "lazy"])
def test_p2_p7_brute_force_dense_emulator(seed, mode_name):
    """[optirs] DormancyDecay moments at touch time equal dense Adam's fed explicit zero
    gradients on dormant steps; no parameter update on dormant steps.  Lazy: single factor.
    Brute force on tiny tables (1-D view of R*c <= 32 coordinates, T <= 20)."""
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 33))
    T = int(rng.integers(1, 21))
    hp = dict(lr=float(rng.choice([1e-3, 1e-2, 0.3])), beta1=float(rng.choice([0.0, 0.5, 0.9])),
              beta2=float(rng.choice([0.0, 0.9, 0.999])), eps=float(rng.choice([1e-8, 1e-3])))
    touches = _random_touches(rng, n, T, float(rng.uniform(0.1, 0.9)))
    p0 = rng.standard_normal(n)
    mode = DD if mode_name == "dormancy_decay" else LAZY
    p, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    ls = np.zeros(n, np.int64)
    emu_state = list(p0)
    for t in range(1, T + 1):
        tch = touches[t - 1]
        idx = np.array(sorted(tch), np.int64)
        g = np.array([tch[i] for i in idx], np.float32)
        assert oracle.adam_step(p, m, v, ls, idx, g, t, mode=mode, **hp) == 0
        ep, em, ev = de.lazy_adam_dense(p0, touches[:t], mode=mode_name, **hp)
        for i in idx:  # at touch time the moments agree (and the parameters)
            assert math.isclose(m[i], em[i], rel_tol=1e-12, abs_tol=1e-300)
            assert math.isclose(v[i], ev[i], rel_tol=1e-12, abs_tol=1e-300)
        np.testing.assert_allclose(p, ep, rtol=1e-12, atol=1e-14)
        emu_state = ep
    assert list(ls) == [max([t for t in range(1, T + 1) if i in touches[t - 1]], default=0)
                        for i in range(n)]


def test_p2_trajectory_differs_from_dense_adam():
    """[optirs] the parameter trajectory differs from dense Adam: lazy Adam performs no
    parameter update on dormant steps."""
    hp = dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8)
    touches = [{0: 1.0}, {}, {0: -0.5}]  # a dormant step at t=2
    lp, lm, lv = de.lazy_adam_dense([0.3], touches, mode="dormancy_decay", **hp)
    dp, dm, dv = de.dense_adam([0.3], touches, **hp)
    assert lm == pytest.approx(dm, rel=1e-15) and lv == pytest.approx(dv, rel=1e-15)
    assert abs(lp[0] - dp[0]) > 1e-6
    p = np.array([0.3])
    m, v, ls = np.zeros(1), np.zeros(1), np.zeros(1, np.int64)
    for t, tch in enumerate(touches, start=1):
        if tch:
            oracle.adam_step(p, m, v, ls, np.array([0]), np.array([tch[0]], np.float32), t,
                             mode=DD, **hp)
    assert p[0] == pytest.approx(lp[0], rel=1e-13)
    assert abs(p[0] - dp[0]) > 1e-6


# --------------------------------------------------------------------------
# P3 / P9: closed form at first touch; bias correction by the global step
# --------------------------------------------------------------------------
@pytest.mark.parametrize("t", [1, 2, 5, 17, 1000])
@pytest.mark.parametrize("mode", [LAZY, DD])
def test_p3_p9_first_touch_closed_form(t, mode):
    """[optirs] with m = v = 0, a first touch at global step t gives m = (1-b1) g,
    v = (1-b2) g^2 and dp = -lr ((1-b1)/(1-b1^t)) g / (|g| sqrt((1-b2)/(1-b2^t)) + eps);
    the bias correction uses t, never the visit count (1)."""
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)
    g = np.array([0.7, -2.5, 1e-3], np.float32)
    p = np.array([0.1, 0.2, -0.3])
    m, v, ls = np.zeros(3), np.zeros(3), np.zeros(3, np.int64)
    ls[:] = 0
    p0 = p.copy()
    assert oracle.adam_step(p, m, v, ls, np.arange(3), g, t, mode=mode, **hp) == 0
    b1, b2, lr, eps = hp["beta1"], hp["beta2"], hp["lr"], hp["eps"]
    gd = g.astype(np.float64)
    want_dp = -lr * ((1 - b1) / (1 - b1 ** t)) * gd / (np.abs(gd) * math.sqrt((1 - b2) / (1 - b2 ** t)) + eps)
    np.testing.assert_allclose(p - p0, want_dp, rtol=1e-10)
    np.testing.assert_allclose(m, (1 - b1) * gd, rtol=1e-15)
    np.testing.assert_allclose(v, (1 - b2) * gd * gd, rtol=1e-15)
    if t > 1:  # a visit-count correction (t = 1) would give a different step
        wrong = -lr * gd / (np.abs(gd) + eps)
        assert np.all(np.abs((p - p0) - wrong) > 1e-6 * np.abs(wrong))
    if t == 1:
        np.testing.assert_allclose(p - p0, -lr * gd / (np.abs(gd) + eps), rtol=1e-10)


# --------------------------------------------------------------------------
# P4: untouched coordinates stay bit-identical
# --------------------------------------------------------------------------
def _canaries(shape, rng):
    a = rng.standard_normal(shape).astype(np.float32)
    flat = a.reshape(-1).view(np.uint32)
    special = np.array([0x7FC01234, 0xFFA00001, 0x80000000, 0x00000001, 0x007FFFFF, 0x7F800000,
                        0xFF800000], np.uint32)
    flat[::3] = special[np.arange(flat[::3].shape[0]) % special.shape[0]]
    return a


@pytest.mark.parametrize("mode", [LAZY, DD])
def test_p4_untouched_bit_identity_rows_and_csr(mode):
    """[optirs] untouched coordinates are left bit-identical (also the other columns of a
    touched row under an element-granular CSR gradient)."""
    rng = np.random.default_rng(5)
    r, c = 12, 6
    p, m, v = (_canaries((r, c), rng) for _ in range(3))
    ls = np.zeros(r * c, np.int64)
    before = [x.copy() for x in (p, m, v)]
    touched = np.zeros((r, c), bool)
    hp = dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8)
    for t in range(1, 6):
        rows = np.sort(rng.choice(r, 4, replace=False))
        row_off = np.zeros(r + 1, np.int64)
        cols = []
        for rr in range(r):
            k = 2 if rr in rows else 0
            cs = np.sort(rng.choice(c, k, replace=False)) if k else np.array([], int)
            cols.extend(cs.tolist())
            touched[rr, cs] = True
            row_off[rr + 1] = row_off[rr] + k
        cols = np.array(cols, np.int32)
        vals = rng.standard_normal(cols.shape[0]).astype(np.float32)
        # touched coordinates must start from valid state: reset those to finite zeros once
        for rr in range(r):
            for j in range(row_off[rr], row_off[rr + 1]):
                if ls[rr * c + cols[j]] == 0:
                    p[rr, cols[j]] = 0.5
                    m[rr, cols[j]] = 0.0
                    v[rr, cols[j]] = 0.0
        assert oracle.adam_table_step(p, m, v, ls, t, row_off=row_off, cols=cols, vals=vals,
                                      ls_per_coord=True, mode=mode, **hp) == 0
    for a, b in zip((p, m, v), before):
        assert a.view(np.uint32)[~touched].tobytes() == b.view(np.uint32)[~touched].tobytes()
        assert np.all(np.isfinite(a[touched]))


def test_p4_sgd_untouched_bit_identity():
    """[optirs] Sparse SGD leaves untouched coordinates (and their buffers) bit-identical."""
    rng = np.random.default_rng(6)
    p = _canaries((50,), rng)
    buf = _canaries((50,), rng)
    idx = np.array([1, 4, 9, 30], np.int64)
    p[idx] = 1.0
    buf[idx] = 0.0
    pb, bb = p.copy(), buf.copy()
    for _ in range(3):
        assert oracle.sgd_step(p, buf, idx, np.ones(4, np.float32), lr=0.1, momentum=0.9,
                               weight_decay=1e-4) == 0
    mask = np.ones(50, bool)
    mask[idx] = False
    assert p[mask].tobytes() == pb[mask].tobytes() and buf[mask].tobytes() == bb[mask].tobytes()


# --------------------------------------------------------------------------
# P5: summed duplicates == pre-aggregated gradient
# --------------------------------------------------------------------------
@pytest.mark.parametrize("mode", [LAZY, DD])
def test_p5_duplicates_equal_preaggregated(mode):
    """[DSA] duplicate indices are summed: a step on raw duplicated COO equals, bit for bit,
    a step on the pre-summed canonical COO (dyadic values: every sum is exact)."""
    rng = np.random.default_rng(7)
    r, c = 40, 3
    hp = dict(lr=1e-2, beta1=0.9, beta2=0.99, eps=1e-8)
    pa = rng.standard_normal((r, c)).astype(np.float32)
    ma, va = np.zeros_like(pa), np.zeros_like(pa)
    pb, mb, vb = pa.copy(), ma.copy(), va.copy()
    lsa, lsb = np.zeros(r, np.int64), np.zeros(r, np.int64)
    for t in range(1, 8):
        rows = rng.integers(0, r, 60)
        vals = (rng.integers(-64, 64, (60, c)) / 16.0).astype(np.float32)
        agg = {}
        for i, rr in enumerate(rows):
            agg.setdefault(int(rr), np.zeros(c))
            agg[int(rr)] += vals[i]
        crow = np.array(sorted(agg), np.int64)
        cval = np.array([agg[k] for k in crow], np.float32)
        assert oracle.adam_table_step(pa, ma, va, lsa, t, rows=rows, vals=vals, mode=mode, **hp) == 0
        assert oracle.adam_table_step(pb, mb, vb, lsb, t, rows=crow, vals=cval, is_canonical=True,
                                      mode=mode, **hp) == 0
    for a, b in ((pa, pb), (ma, mb), (va, vb), (lsa, lsb)):
        assert a.tobytes() == b.tobytes()


def test_canonicalize_brute_force():
    """[DSA] duplicates summed and sorted after dedup: brute force with a dict on small raw
    inputs; values summed in input order in fp64 and rounded once (a lone value unchanged)."""
    rng = np.random.default_rng(8)
    for trial in range(30):
        n = int(rng.integers(0, 200))
        bound = int(rng.integers(1, 50))
        c = int(rng.integers(1, 5))
        idx = rng.integers(0, bound, n)
        vals = rng.standard_normal((n, c)).astype(np.float32)
        if n:
            vals[rng.integers(0, n)] = -0.0
        groups = {}
        for i in range(n):
            groups.setdefault(int(idx[i]), []).append(i)
        keys = sorted(groups)
        want_v = np.array([[float(sum_in_order(vals[groups[k], j])) for j in range(c)] for k in keys],
                          np.float64).astype(np.float32).reshape(-1, c)
        ci, cv, seg, perm = oracle.canonicalize(idx, vals, bound)
        assert list(ci) == keys
        assert cv.reshape(-1, c).tobytes() == want_v.tobytes()
        assert list(np.diff(seg)) == [len(groups[k]) for k in keys]
        assert list(perm) == [i for k in keys for i in groups[k]]


def sum_in_order(xs):
    s = float(xs[0])
    for x in xs[1:]:
        s += float(x)
    return s


# --------------------------------------------------------------------------
# P6: CSR <-> COO round trips
# --------------------------------------------------------------------------
def test_p6_round_trips():
    """[optirs] CsrGradient::to_coo / from_coo are lossless; COO from CSR is strictly ascending."""
    rng = np.random.default_rng(9)
    for trial in range(40):
        r = int(rng.integers(0, 30))
        c = int(rng.integers(1, 12))
        k = int(rng.integers(0, r * c + 1)) if r else 0
        lin = np.sort(rng.choice(r * c, size=k, replace=False)).astype(np.int64) if r else np.zeros(0, np.int64)
        ro, co = oracle.coo_to_csr(lin, r, c)
        assert ro[0] == 0 and ro[-1] == k and np.all(np.diff(ro) >= 0)
        back = oracle.csr_to_coo(ro, co, r, c)
        assert np.array_equal(back, lin)
        assert np.all(np.diff(back) > 0)
        ro2, co2 = oracle.coo_to_csr(back, r, c)
        assert np.array_equal(ro2, ro) and np.array_equal(co2, co)
        # brute force: rows by integer division
        assert np.array_equal(np.repeat(np.arange(r), np.diff(ro)), lin // c)
        assert np.array_equal(co, (lin % c).astype(np.int32))


def test_row_coo_to_csr_full_rows():
    """Canonical row-COO as CSR: every listed row holds all c columns in order."""
    rows = np.array([1, 4, 5], np.int64)
    ro, co = oracle.row_coo_to_csr(rows, 7, 3)
    assert list(ro) == [0, 0, 3, 3, 3, 6, 9, 9]
    assert list(co) == [0, 1, 2] * 3
    assert np.array_equal(oracle.csr_to_coo(ro, co, 7, 3), (rows[:, None] * 3 + np.arange(3)).ravel())


# --------------------------------------------------------------------------
# P8: SGD against the textbook (torch.optim.SGD)
# --------------------------------------------------------------------------
def test_p8_sgd_plain_and_vs_torch():
    """[optirs] Sparse SGD: params[i] -= lr*grad[i] (mu = 0, wd = 0); with every coordinate
    touched every step, momentum and coupled weight decay match torch.optim.SGD (dampening 0)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(10)
    p = rng.standard_normal(20)
    g = rng.standard_normal(20).astype(np.float32)
    p0 = p.copy()
    assert oracle.sgd_step(p, None, np.arange(20), g, lr=0.25, momentum=0.0, weight_decay=0.0) == 0
    assert np.array_equal(p, p0 - 0.25 * g.astype(np.float64))
    r, c, T = 4, 5, 15
    hp = dict(lr=0.05, momentum=0.9, weight_decay=1e-4)
    p0 = rng.standard_normal((r, c))
    grads = rng.standard_normal((T, r, c)).astype(np.float32)
    p, buf = p0.copy(), np.zeros((r, c))
    for t in range(T):
        assert oracle.sgd_table_step(p, buf, rows=np.arange(r), vals=grads[t], is_canonical=True, **hp) == 0
    tp = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.SGD([tp], lr=hp["lr"], momentum=hp["momentum"], dampening=0.0,
                          weight_decay=hp["weight_decay"], foreach=False)
    for t in range(T):
        tp.grad = torch.tensor(grads[t].astype(np.float64))
        opt.step()
    np.testing.assert_allclose(p, tp.detach().numpy(), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(buf, opt.state[tp]["momentum_buffer"].numpy(), rtol=1e-13, atol=1e-15)


def test_sgd_brute_force_dense_emulator():
    """[optirs] lazy momentum on touched coordinates only: oracle == dense emulator loop."""
    rng = np.random.default_rng(12)
    for seed in range(5):
        n, T = 16, 12
        touches = _random_touches(rng, n, T, 0.4)
        hp = dict(lr=0.1, momentum=0.9, weight_decay=1e-2)
        p0 = rng.standard_normal(n)
        p, buf = p0.copy(), np.zeros(n)
        for t in range(T):
            idx = np.array(sorted(touches[t]), np.int64)
            g = np.array([touches[t][i] for i in idx], np.float32)
            assert oracle.sgd_step(p, buf, idx, g, **hp) == 0
        ep, eb = de.sparse_sgd_dense(p0, touches, **hp)
        np.testing.assert_allclose(p, ep, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(buf, eb, rtol=1e-13, atol=1e-15)


# --------------------------------------------------------------------------
# error behaviour: validate before writing anything
# --------------------------------------------------------------------------
def test_errors_leave_state_untouched():
    """[DSA] Validated Inputs: negative / out-of-range indices are explicit errors; the
    step is rejected before anything is written."""
    rng = np.random.default_rng(13)
    r, c = 10, 2
    hp = dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8, mode=DD)
    p = rng.standard_normal((r, c)).astype(np.float32)
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    ls = np.zeros(r, np.int64)
    ls[3] = 5
    snap = [a.copy() for a in (p, m, v, ls)]
    g = np.ones((2, c), np.float32)
    cases = [
        (dict(rows=np.array([1, 10]), vals=g), oracle.ERR_INDEX_OUT_OF_RANGE),
        (dict(rows=np.array([-1, 2]), vals=g), oracle.ERR_INDEX_OUT_OF_RANGE),
        (dict(rows=np.array([2, 2]), vals=g, is_canonical=True), oracle.ERR_NOT_CANONICAL),
        (dict(rows=np.array([4, 2]), vals=g, is_canonical=True), oracle.ERR_NOT_CANONICAL),
        (dict(rows=np.array([3, 4]), vals=g), oracle.ERR_STEP_ORDER),  # t = 5 <= last_step[3]
        (dict(row_off=np.array([0, 1] + [1] * 9, np.int64), cols=np.array([0], np.int32),
              vals=np.ones(1, np.float32)), oracle.ERR_NOT_CANONICAL),  # per-row ls: partial row
        (dict(row_off=np.array([0, 2] + [2] * 9, np.int64), cols=np.array([1, 0], np.int32),
              vals=np.ones(2, np.float32)), oracle.ERR_NOT_CANONICAL),
        (dict(row_off=np.array([0, 1] + [1] * 9, np.int64), cols=np.array([2], np.int32),
              vals=np.ones(1, np.float32)), oracle.ERR_INDEX_OUT_OF_RANGE),
    ]
    for kw, want in cases:
        assert oracle.adam_table_step(p, m, v, ls, 5, **hp, **kw) == want, kw
        for a, b in zip((p, m, v, ls), snap):
            assert a.tobytes() == b.tobytes()
    assert oracle.adam_table_step(p, m, v, ls, 0, rows=np.array([1]), vals=g[:1], **hp) == oracle.ERR_INVALID_ARG
    bad = dict(hp, beta1=1.0)
    assert oracle.adam_table_step(p, m, v, ls, 6, rows=np.array([1]), vals=g[:1], **bad) == oracle.ERR_INVALID_ARG
    assert oracle.canonicalize(np.array([0, 7]), np.ones(2, np.float32), 7, check=False) == 2
    assert oracle.coo_to_csr(np.array([3, 3]), 2, 4, check=False) == 3
    assert oracle.coo_to_csr(np.array([8]), 2, 4, check=False) == 2


def test_zero_work_is_noop():
    """nnz = 0: a legal step that changes nothing."""
    p = np.arange(6, dtype=np.float32).reshape(3, 2)
    m, v = np.zeros_like(p), np.zeros_like(p)
    ls = np.zeros(3, np.int64)
    snap = p.copy()
    assert oracle.adam_table_step(p, m, v, ls, 1, rows=np.zeros(0, np.int64), vals=np.zeros((0, 2), np.float32),
                                  lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, mode=DD) == 0
    assert p.tobytes() == snap.tobytes() and not ls.any()


# --------------------------------------------------------------------------
# P11: row gather (DSA README, read_rows)
# --------------------------------------------------------------------------
def test_p11_read_rows_equals_fancy_indexing_bitwise():
    """The gather is numpy fancy indexing, bit for bit (NaN payloads, -0.0, denormals)."""
    rng = np.random.default_rng(21)
    t = rng.standard_normal((50, 7)).astype(np.float32)
    t.view(np.uint32)[3, 2] = 0x7FC01234          # a NaN with a payload
    t[4, 0], t[4, 1] = np.float32(-0.0), np.float32(1e-42)
    idx = rng.integers(0, 50, 300)
    idx[:4] = [3, 4, 49, 0]
    got = oracle.read_rows(t, idx)
    assert got.tobytes() == t[idx].tobytes()
    assert oracle.read_rows(t, np.zeros(0, np.int64)).shape == (0, 7)
    one_d = rng.standard_normal(9).astype(np.float32)
    assert oracle.read_rows(one_d, np.array([8, 1])).reshape(-1).tobytes() == one_d[[8, 1]].tobytes()


def test_p11_read_rows_rejects_bad_indices():
    t = np.zeros((5, 2), np.float32)
    assert oracle.read_rows(t, np.array([0, 5]), check=False) == oracle.ERR_INDEX_OUT_OF_RANGE
    assert oracle.read_rows(t, np.array([-1]), check=False) == oracle.ERR_INDEX_OUT_OF_RANGE


# --------------------------------------------------------------------------
# P12: non-finite gradients (DSA README, "Validated Inputs")
# --------------------------------------------------------------------------
def test_p12_check_finite():
    rng = np.random.default_rng(31)
    g = rng.standard_normal((100, 8)).astype(np.float32)
    g[7, 3] = np.float32(3.4e38)                 # large but finite
    g[8, 1] = np.float32(1e-45)                  # denormal
    assert oracle.check_finite(g) == oracle.OK
    assert oracle.check_finite(np.zeros(0, np.float32)) == oracle.OK
    for bad in (np.nan, np.inf, -np.inf):
        h = g.copy()
        h[99, 7] = bad
        assert oracle.check_finite(h) == oracle.ERR_NON_FINITE
        assert oracle.check_finite(h) == (oracle.ERR_NON_FINITE if not np.isfinite(h).all() else oracle.OK)


# --------------------------------------------------------------------------
# P13: corrupted moment state (DSA README, "Validated Inputs": NaN / negative
# moment rows).  Pinned against numpy's isfinite and comparison on the gathered
# coordinates, over random tables with planted specials (brute force).
# --------------------------------------------------------------------------
_SPECIALS = [np.nan, np.inf, -np.inf, -1e-3, -1e-42, -0.0, 1e-42, 0.0]


def _numpy_state_ok(m, v, rows=None, row_off=None, cols=None):
    if row_off is not None:
        rr = np.repeat(np.arange(m.shape[0]), np.diff(row_off))
        mt, vt = m[rr, cols], v[rr, cols]
    else:
        mt, vt = m[rows], v[rows]
    return bool(np.isfinite(mt).all() and np.isfinite(vt).all() and (vt >= 0).all())


def test_p13_check_state_matches_numpy_brute_force():
    rng = np.random.default_rng(41)
    seen = {oracle.OK: 0, oracle.ERR_BAD_STATE: 0}
    for trial in range(400):
        r, c = int(rng.integers(1, 9)), int(rng.integers(1, 5))
        m = rng.standard_normal((r, c)).astype(np.float32)
        v = np.abs(rng.standard_normal((r, c))).astype(np.float32)
        for _ in range(int(rng.integers(0, 3))):
            arr = m if rng.random() < 0.5 else v
            arr[rng.integers(0, r), rng.integers(0, c)] = _SPECIALS[rng.integers(0, len(_SPECIALS))]
        if trial % 2 == 0:
            rows = rng.integers(0, r, int(rng.integers(0, 6)))
            got = oracle.check_state(m, v, rows=rows)
            ok = _numpy_state_ok(m, v, rows=rows)
        else:
            counts = rng.integers(0, c + 1, r)
            row_off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
            cols = np.concatenate([np.sort(rng.choice(c, k, replace=False)) for k in counts]).astype(np.int32) \
                if counts.sum() else np.zeros(0, np.int32)
            got = oracle.check_state(m, v, row_off=row_off, cols=cols)
            ok = _numpy_state_ok(m, v, row_off=row_off, cols=cols)
        assert got == (oracle.OK if ok else oracle.ERR_BAD_STATE), (trial, got, ok)
        seen[got] += 1
    assert seen[oracle.OK] > 50 and seen[oracle.ERR_BAD_STATE] > 50


def test_p13_check_state_cases():
    m = np.zeros((4, 3), np.float32)
    v = np.zeros((4, 3), np.float32)
    v[1, 2] = np.float32(-0.0)                     # -0.0 is not below zero
    m[2, 0] = np.float32(-1e-42)                   # a negative first moment is legal
    assert oracle.check_state(m, v, rows=np.array([1, 2, 1])) == oracle.OK
    v[3, 1] = np.float32(-1e-45)                   # the smallest negative v
    assert oracle.check_state(m, v, rows=np.array([0, 1, 2])) == oracle.OK   # row 3 untouched
    assert oracle.check_state(m, v, rows=np.array([3])) == oracle.ERR_BAD_STATE
    # CSR: only the listed columns of a row are read
    row_off = np.array([0, 0, 0, 0, 2], np.int64)
    assert oracle.check_state(m, v, row_off=row_off, cols=np.array([0, 2], np.int32)) == oracle.OK
    assert oracle.check_state(m, v, row_off=row_off, cols=np.array([1, 2], np.int32)) == oracle.ERR_BAD_STATE
    m[0, 1] = np.float32(np.inf)
    assert oracle.check_state(m, v, rows=np.array([0])) == oracle.ERR_BAD_STATE
    assert oracle.check_state(m, v, rows=np.array([4])) == oracle.ERR_INDEX_OUT_OF_RANGE
    assert oracle.check_state(m, v, rows=np.array([-1])) == oracle.ERR_INDEX_OUT_OF_RANGE
    assert oracle.check_state(m, v, rows=np.zeros(0, np.int64)) == oracle.OK
    # 1-D parameter
    m1, v1 = np.zeros(5, np.float32), np.ones(5, np.float32)
    v1[4] = np.nan
    assert oracle.check_state(m1, v1, rows=np.array([0, 3])) == oracle.OK
    assert oracle.check_state(m1, v1, rows=np.array([4])) == oracle.ERR_BAD_STATE
