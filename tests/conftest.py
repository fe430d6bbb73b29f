import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Near-tie tokens of every GPU parity comparison, reported separately
    from the pass/fail result (their routing is checked against the oracle
    recomputed with the GPU's ids instead)."""
    mod = sys.modules.get("gpu_harness")
    reps = getattr(mod, "REPORTS", None) if mod else None
    if not reps:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity comparisons: near ties reported separately")
    for r in reps:
        tr.write_line(f"{r['test']}: tokens {r['tokens']}, rows compared {r['rows_compared']}, "
                      f"near ties {r['near_ties']}, worst err/bound {r['worst_ratio']:.3f}")
    tr.write_line(f"total near-tie tokens: {sum(r['near_ties'] for r in reps)} "
                  f"over {sum(r['tokens'] for r in reps)} routed tokens")
