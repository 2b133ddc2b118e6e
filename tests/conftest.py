import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs on the GB300)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def repo_root():
    return ROOT


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Near-tie counts and errors of every GPU parity check of the session."""
    mod = sys.modules.get("parity_util")
    if mod is None or not getattr(mod, "REPORTS", None):
        return
    terminalreporter.write_sep("-", "parity near-tie counts (count / denominator)")
    for line in mod.summary_lines():
        terminalreporter.write_line(line)
