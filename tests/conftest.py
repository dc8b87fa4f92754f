import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size parity case")


def pytest_terminal_summary(terminalreporter):
    """Worst max-abs error next to its bound per workload and tensor, for every
    comparison the parity helpers made in this run."""
    parity = sys.modules.get("parity")
    if parity is None or not getattr(parity, "RECORDS", None):
        return
    terminalreporter.section("max-abs error / bound per workload and tensor")
    for line in parity.summary_lines():
        terminalreporter.line(line)
