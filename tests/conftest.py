import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Worst per-token error (the asserted bar) and worst element-wise error
    |y - y_ref| / max(|y_ref|, 1e-3 rms(y_ref)) (a diagnostic) of every parity
    check that ran, by test case."""
    diag = sys.modules.get("parity_util")
    diag = getattr(diag, "DIAG", None)
    if not diag:
        return
    tr = terminalreporter
    tr.section("parity against the oracle: worst per-token / element-wise relative error")
    for key in sorted(diag):
        tok, elem = diag[key]
        tr.write_line(f"{tok:10.3e} {elem:10.3e}  {key}")
