import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def pytest_terminal_summary(terminalreporter):
    """Achieved parity margins of every oracle comparison that ran."""
    gu = sys.modules.get("gpu_util")
    rows = getattr(gu, "MARGINS", None)
    if not rows:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity margins against the fp64 oracle (bound: max-abs 1e-2, max-rel 1e-2)")
    worst_abs = max(r[2] for r in rows if r[1] != "lse")
    worst_rel = max(r[3] for r in rows if r[1] != "lse")
    for test, what, max_abs, max_rel, n in rows:
        tr.write_line(f"{test} [{what}] max-abs {max_abs:.3e} max-rel {max_rel:.3e} n={n}")
    tr.write_line(f"worst over {len(rows)} comparisons: max-abs {worst_abs:.3e}, max-rel {worst_rel:.3e}")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle.build()
    return oracle
