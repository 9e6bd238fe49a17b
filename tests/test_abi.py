"""The C-ABI library loads and exports every entry point include/sparseopt.h declares (no GPU)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "sparseopt.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sparse_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib_path():
    from lazy_optimizers_embedding_gb300 import build
    return build.build()


def test_header_declares_the_hot_path():
    names = declared_functions()
    for want in ("sparse_canonicalize", "sparse_adam_step", "sparse_adam_table_step", "sparse_sgd_step",
                 "sparse_sgd_table_step", "sparse_csr_to_coo", "sparse_coo_to_csr", "sparse_workspace_size",
                 "sparse_status_string"):
        assert want in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol(lib_path):
    from lazy_optimizers_embedding_gb300 import binding
    assert set(declared_functions()) == set(binding.EXPORTED)
    for n in binding.EXPORTED:
        assert callable(getattr(binding, n))


def test_host_side_queries(lib_path):
    from lazy_optimizers_embedding_gb300 import binding as so
    assert so.status_string(so.OK) == "ok"
    assert "range" in so.status_string(so.ERR_INDEX_OUT_OF_RANGE)
    assert so.status_string(99) == "unknown status"
    small = so.sparse_workspace_size(1000, 64, 10_000)
    big = so.sparse_workspace_size(262_144, 128, 10_000_000)
    assert 0 < small < big
    # workspace grows about linearly in n (keys, positions, pieces, partial slots)
    assert big < 262_144 * (4 * 4 + 16 + 4 + 2 * 2 * 128 * 4 / 32 * 2 + 64)
    assert so.sparse_workspace_size(-1, 1, 1) == 0


def test_row_count_limits_rejected_on_the_host(lib_path):
    """Row-COO tables of more than 2^32 rows are refused before anything is enqueued (raw keys
    and the rows of a canonical table are 32-bit inside the library); the pointers are never
    dereferenced, so placeholders serve."""
    import ctypes
    from lazy_optimizers_embedding_gb300 import binding as so
    fake = ctypes.c_void_p(256)
    cfg = so.AdamConfig(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)
    for canonical in (0, 1):
        g = so.Grad(form=so.GRAD_ROW_COO, n=4, row_idx=256, vals=256, is_canonical=canonical)
        rc = so.LIB.sparse_adam_table_step(fake, fake, fake, fake, so.LAST_STEP_PER_ROW, (1 << 32) + 1, 1,
                                           ctypes.byref(g), 1, cfg, so.DORMANCY_DECAY, fake, 1 << 20, fake, None)
        assert rc == so.ERR_INVALID_ARG
