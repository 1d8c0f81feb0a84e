import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running (full-size workloads)")


_PARITY = []


@pytest.fixture
def parity_report():
    """Records per-tensor parity errors of a case; they are printed at the end of the run."""

    def add(case, errs):
        _PARITY.append((case, errs))

    return add


def pytest_terminal_summary(terminalreporter):
    if not _PARITY:
        return
    terminalreporter.section("parity against the fp64 oracle (relative L2, max-abs / max|ref|)")
    for case, errs in _PARITY:
        parts = [f"{k} {v['rel_l2']:.2e} {v['max_abs_frac']:.2e}" for k, v in errs.items()]
        terminalreporter.write_line(f"{case}: " + "; ".join(parts))
