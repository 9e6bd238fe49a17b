"""Seeded input generators: deterministic, and shaped like the specified workloads."""
import numpy as np

from lazy_optimizers_embedding_gb300 import workloads as wl


def test_steps_are_reproducible_and_distinct():
    w = wl.CFG_ZIPF_10M_128.scaled(rows=100_000, lookups=4096)
    a_idx, a_val = wl.coo_step(w, 3)
    b_idx, b_val = wl.coo_step(w, 3)
    c_idx, _ = wl.coo_step(w, 4)
    assert np.array_equal(a_idx, b_idx) and a_val.tobytes() == b_val.tobytes()
    assert not np.array_equal(a_idx, c_idx)
    assert a_idx.dtype == np.int64 and a_val.dtype == np.float32 and a_val.shape == (4096, 128)
    assert a_idx.min() >= 0 and a_idx.max() < w.rows


def test_zipf_head_mass():
    """Bounded Zipf(s): P(row 0) = 1 / H_N(s)."""
    w = wl.CFG_ZIPF_1M_64.scaled(rows=50_000, lookups=200_000)
    idx, _ = wl.coo_step(w, 0)
    h = np.sum(np.arange(1, w.rows + 1, dtype=np.float64) ** -w.zipf_s)
    frac0 = np.mean(idx == 0)
    assert abs(frac0 - 1 / h) < 5 * np.sqrt((1 / h) / len(idx))


def test_table_init_subset_matches_full():
    w = wl.CFG_CSR_4M_256.scaled(rows=200_000, cols=8)
    full = wl.table_init(w)
    rows = np.array([0, 65535, 65536, 199_999, 12345])
    assert full[rows].tobytes() == wl.table_init(w, rows).tobytes()
    assert abs(full.std() - w.init_std) < 1e-3 * 5


def test_csr_elem_shape():
    w = wl.CFG_CSR_4M_256.scaled(rows=10_000, lookups=500)
    row_off, cols, vals = wl.csr_elem_step(w, 0)
    assert row_off.shape == (w.rows + 1,) and row_off[-1] == 500 * 16 == cols.shape[0] == vals.shape[0]
    per_row = np.diff(row_off)
    assert set(np.unique(per_row)) <= {0, 16} and (per_row == 16).sum() == 500
    c2 = cols.reshape(-1, 16)
    assert np.all(np.diff(c2, axis=1) > 0) and c2.min() >= 0 and c2.max() < w.cols


def test_unique_sorted_1d():
    idx, g = wl.coo_step(wl.CFG_1D, 0)
    assert idx.shape == (1000,) and np.all(np.diff(idx) > 0) and g.shape == (1000, 1)
