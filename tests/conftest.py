import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload; minutes on the host side")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """Index mismatches and near-boundary draws of the GPU parity tests, by configuration
    (printed when any batch was compared in this run)."""
    helpers = sys.modules.get("tests.gpu_helpers")
    counts = getattr(helpers, "BOUNDARY_COUNTS", None)
    if not counts:
        return
    tr = terminalreporter
    tr.section("boundary draws (index mismatches must be near-boundary draws, < 0.01% of draws)")
    for name in sorted(counts):
        c = counts[name]
        frac = c["mismatch"] / c["draws"] if c["draws"] else 0.0
        tr.write_line(f"{name}: draws {c['draws']}, mismatch {c['mismatch']} ({100 * frac:.5f}%), "
                      f"near-boundary {c['near']} ({100 * c['near'] / max(c['draws'], 1):.3f}%)")
