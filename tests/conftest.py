import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Prints the near-tie counts the parity tests recorded: decisions where the GPU's
    choice differs from the oracle's own but lies within the 1e-4 margin (accepted)."""
    try:
        import parity
    except ImportError:
        return
    if not parity.REPORTS:
        return
    terminalreporter.write_sep("-", "accepted near-tie decisions (GPU choice != oracle's, within the 1e-4 margin)")
    for what, counts in parity.REPORTS:
        terminalreporter.write_line(f"{what}: " + ", ".join(f"{k}={v}" for k, v in counts.items()))
