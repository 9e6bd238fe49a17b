"""Seeded synthetic inputs for the sparse / lazy optimizer step.

This module only *draws* inputs: row indices, gradient values and initial table
values.  It holds none of the optimizer's arithmetic (no duplicate summing, no
sorting into canonical form beyond what a workload defines as its input, no
optimizer math), so that the CPU oracle and the CUDA path can both be fed from
it without sharing any computation.

Every stream is a numpy PCG64 generator keyed by ``SeedSequence([seed, stream,
k])``: ``stream`` separates index draws, value draws and table initialisation,
``k`` is the step (or the 65,536-row block of the table), so any step or any
table block can be regenerated on its own, on any machine, bit for bit.

The five workloads are the embedding-table shapes the sparse optimizer step is
specified on: a 1-D parameter touched at unique ascending coordinates, Zipf- and
uniform-indexed lookups into 2-D tables (raw COO with duplicates), and an
element-granular CSR gradient.  Zipf(s) over N rows is the bounded Zipf law
P(rank k) proportional to k**-s, k = 1..N, with rank k mapped to row k-1.
"""
from __future__ import annotations

import dataclasses
import functools
from concurrent.futures import ThreadPoolExecutor

import numpy as np

STREAM_INDEX = 1
STREAM_VALUES = 2
STREAM_INIT = 3
STREAM_COLS = 4
INIT_BLOCK_ROWS = 65536


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and value distributions of one synthetic workload.

    ``index_dist`` is one of
      * ``"unique_sorted"`` - ``lookups`` distinct rows drawn uniformly without
        replacement, strictly ascending (a canonical COO gradient);
      * ``"zipf"``          - ``lookups`` rows drawn i.i.d. from bounded Zipf(``zipf_s``),
        unsorted, duplicates allowed (a raw COO gradient);
      * ``"uniform"``       - ``lookups`` rows drawn i.i.d. uniformly (raw COO);
      * ``"csr_elem"``      - ``lookups`` distinct rows drawn uniformly, each with
        ``csr_cols_per_row`` distinct ascending columns (an element-granular CSR).
    Gradient values are N(0, grad_std**2); the table starts N(0, init_std**2).
    """

    name: str
    rows: int
    cols: int
    steps: int
    lookups: int
    index_dist: str
    grad_std: float
    init_std: float
    zipf_s: float = 0.0
    csr_cols_per_row: int = 0
    optimizer: str = "adam"            # "adam" | "sgd"
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    momentum: float = 0.0
    weight_decay: float = 0.0
    seed: int = 0

    def scaled(self, **kw) -> "Workload":
        """Same distributions at other sizes (for parity cases the oracle finishes quickly)."""
        return dataclasses.replace(self, **kw)

    @property
    def coords(self) -> int:
        return self.rows * self.cols


# The five specified workloads (sizes exactly as specified).
CFG_1D = Workload("1d_100k_unique1000", rows=100_000, cols=1, steps=10, lookups=1_000,
                  index_dist="unique_sorted", grad_std=1.0, init_std=1.0)
CFG_1D_SGD = CFG_1D.scaled(name="1d_100k_unique1000_sgd", optimizer="sgd", lr=1e-2, momentum=0.9)
CFG_ZIPF_1M_64 = Workload("table_1Mx64_zipf1.1_csr", rows=1_000_000, cols=64, steps=100,
                          lookups=65_536, index_dist="zipf", zipf_s=1.1,
                          grad_std=1e-2, init_std=1e-2)
CFG_ZIPF_10M_128 = Workload("table_10Mx128_zipf1.05_coo", rows=10_000_000, cols=128, steps=50,
                            lookups=262_144, index_dist="zipf", zipf_s=1.05,
                            grad_std=1e-2, init_std=1e-2)
CFG_CSR_4M_256 = Workload("table_4Mx256_csr131072x16", rows=4_000_000, cols=256, steps=50,
                          lookups=131_072, index_dist="csr_elem", csr_cols_per_row=16,
                          grad_std=1.0, init_std=1e-2)
CFG_SGD_50M_32 = Workload("table_50Mx32_uniform_sgd", rows=50_000_000, cols=32, steps=20,
                          lookups=1_048_576, index_dist="uniform", grad_std=1.0, init_std=1e-2,
                          optimizer="sgd", lr=0.05, momentum=0.9, weight_decay=1e-4)

ALL = (CFG_1D, CFG_1D_SGD, CFG_ZIPF_1M_64, CFG_ZIPF_10M_128, CFG_CSR_4M_256, CFG_SGD_50M_32)


def rng(seed: int, stream: int, k: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, k])))


@functools.lru_cache(maxsize=4)
def _zipf_cdf(n_rows: int, s: float) -> np.ndarray:
    weights = np.arange(1, n_rows + 1, dtype=np.float64) ** (-s)
    return np.cumsum(weights)


def zipf_rows(g: np.random.Generator, n: int, n_rows: int, s: float) -> np.ndarray:
    """i.i.d. draws of bounded Zipf(s) over ``n_rows`` rows (rank k -> row k-1), by inverse CDF."""
    cdf = _zipf_cdf(n_rows, s)
    u = g.random(n) * cdf[-1]
    r = np.searchsorted(cdf, u, side="right")
    return np.minimum(r, n_rows - 1).astype(np.int64)


def step_indices(w: Workload, step: int) -> np.ndarray:
    """Row (or 1-D coordinate) indices of one step; for ``csr_elem`` the touched rows."""
    g = rng(w.seed, STREAM_INDEX, step)
    if w.index_dist == "zipf":
        return zipf_rows(g, w.lookups, w.rows, w.zipf_s)
    if w.index_dist == "uniform":
        return g.integers(0, w.rows, size=w.lookups, dtype=np.int64)
    if w.index_dist in ("unique_sorted", "csr_elem"):
        idx = g.choice(w.rows, size=w.lookups, replace=False, shuffle=False).astype(np.int64)
        idx.sort()
        return idx
    raise ValueError(w.index_dist)


def step_values(w: Workload, step: int, n: int) -> np.ndarray:
    """``n`` gradient values (or rows of ``cols`` values) of one step, N(0, grad_std**2), fp32."""
    g = rng(w.seed, STREAM_VALUES, step)
    shape = (n,) if w.index_dist == "csr_elem" else (n, w.cols)
    z = g.standard_normal(shape, dtype=np.float32)
    z *= np.float32(w.grad_std)
    return z


def coo_step(w: Workload, step: int):
    """(indices int64[n], values fp32[n, cols]) of one COO step (raw or canonical per the workload)."""
    idx = step_indices(w, step)
    return idx, step_values(w, step, idx.shape[0])


def csr_elem_step(w: Workload, step: int):
    """(row_off int64[rows+1], cols int32[nnz], values fp32[nnz]) of one element-granular CSR step.

    Touched rows are distinct and uniform; within each, ``csr_cols_per_row`` distinct columns are
    chosen uniformly and listed in ascending order.  Offsets are the running count of listed
    entries per row over all ``rows`` rows (empty rows included).
    """
    assert w.index_dist == "csr_elem"
    rows = step_indices(w, step)
    k = w.csr_cols_per_row
    g = rng(w.seed, STREAM_COLS, step)
    keys = g.random((rows.shape[0], w.cols), dtype=np.float32)
    sel = np.argpartition(keys, k - 1, axis=1)[:, :k] if k < w.cols else np.tile(
        np.arange(w.cols), (rows.shape[0], 1))
    sel = np.sort(sel, axis=1).astype(np.int32)
    counts = np.zeros(w.rows, dtype=np.int64)
    counts[rows] = k
    row_off = np.zeros(w.rows + 1, dtype=np.int64)
    np.cumsum(counts, out=row_off[1:])
    vals = step_values(w, step, rows.shape[0] * k)
    return row_off, sel.reshape(-1), vals


def _init_block(w: Workload, b: int) -> np.ndarray:
    lo = b * INIT_BLOCK_ROWS
    hi = min(w.rows, lo + INIT_BLOCK_ROWS)
    z = rng(w.seed, STREAM_INIT, b).standard_normal((hi - lo, w.cols), dtype=np.float32)
    z *= np.float32(w.init_std)
    return z


def table_init(w: Workload, rows: np.ndarray | None = None, threads: int = 8) -> np.ndarray:
    """Initial table, fp32 [rows, cols] (or only the listed ``rows``), N(0, init_std**2).

    Generated in blocks of 65,536 rows, each from its own stream, so a subset of rows is
    reproducible without drawing the whole table.
    """
    if rows is None:
        out = np.empty((w.rows, w.cols), dtype=np.float32)
        nb = (w.rows + INIT_BLOCK_ROWS - 1) // INIT_BLOCK_ROWS

        def fill(b):
            lo = b * INIT_BLOCK_ROWS
            blk = _init_block(w, b)
            out[lo:lo + blk.shape[0]] = blk

        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(fill, range(nb)))
        return out
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((rows.shape[0], w.cols), dtype=np.float32)
    blocks = rows // INIT_BLOCK_ROWS
    for b in np.unique(blocks):
        blk = _init_block(w, int(b))
        sel = np.nonzero(blocks == b)[0]
        out[sel] = blk[rows[sel] - b * INIT_BLOCK_ROWS]
    return out


def coo_steps_parallel(w: Workload, steps, threads: int = 8):
    """``coo_step`` for several steps, drawn on a thread pool (numpy releases the GIL)."""
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda s: coo_step(w, s), steps))
