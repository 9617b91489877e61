import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_terminal_summary(terminalreporter):
    try:
        from tests.gpu_util import PARITY_LOG
    except Exception:
        return
    if not PARITY_LOG:
        return
    terminalreporter.write_sep("-", "layer-output parity (rel_l2, max_abs/rms) vs the oracle")
    for name, rel, mx in PARITY_LOG:
        terminalreporter.write_line(f"{name:40s} rel_l2={rel:.3e} max_abs/rms={mx:.3e}")
