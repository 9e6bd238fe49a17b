import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


def read_cases(name):
    """Parse a golden fixture: '#' comments, 'case' separators, 'key v1 v2 ...' lines."""
    cases, cur = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line == "case":
                if cur:
                    cases.append(cur)
                cur = {}
                continue
            key, *vals = line.split()
            cur.setdefault(key, []).append(vals)
    if cur:
        cases.append(cur)
    return cases


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library through its Python binding; skips when no GPU is present."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from lazy_optimizers_embedding_gb300 import binding
    return binding


def pytest_terminal_summary(terminalreporter):
    """The largest no-floor moment errors the GPU parity tests measured (see gpu_harness)."""
    h = sys.modules.get("gpu_harness")
    if h is None or not getattr(h, "DIAG", None):
        return
    terminalreporter.section("parity diagnostics (largest errors seen)")
    for key in sorted(h.DIAG):
        vals = ", ".join(f"{q} {v:.3e}" for q, v in sorted(h.DIAG[key].items()))
        terminalreporter.write_line(f"{key}: {vals}")
