import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long CPU test")


def pytest_terminal_summary(terminalreporter):
    """The K/V ulp histogram of the GPU parity checks that ran (if any)."""
    h = sys.modules.get("harness")
    if h is not None and h.KV_STATS["elements"]:
        terminalreporter.write_line(h.kv_stats_line())
