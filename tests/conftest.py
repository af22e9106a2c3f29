import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """The near-tie exclusions of the GPU comparisons, per workload and rule: requests
    compared, identical to the oracle, and left out on each rule (with the oracle's own
    near-tie counts beside them)."""
    from parity import REPORT
    if not REPORT:
        return
    tr = terminalreporter
    tr.write_sep("-", "near-tie exclusions (GPU vs oracle)")
    for name, t in REPORT:
        ex = " ".join(f"{r}={t['excluded'][r]}" for r in t["excluded"])
        near = " ".join(f"{r}={t['near'][r]}" for r in t["near"])
        tr.write_line(f"{name}: {t['exact']}/{t['requests']} identical; excluded {ex}; "
                      f"oracle near-ties {near}")
