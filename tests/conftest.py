import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a) and the built CUDA library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """After a run of the GPU parity tests: how much of the oracle's near-tie slack each
    comparison used (see gpu_helpers)."""
    helpers = sys.modules.get("gpu_helpers")
    if helpers is not None:
        for line in helpers.slack_table():
            terminalreporter.write_line(line)
    bwd = sys.modules.get("test_gpu_backward") or sys.modules.get("tests.test_gpu_backward")
    if bwd is not None and bwd.RATIO_LOG:
        terminalreporter.write_line("backward parity: largest |gpu - oracle| / bound per case (dq, dk, dv)")
        for name, rq, rk, rv in bwd.RATIO_LOG:
            terminalreporter.write_line(f"  {name:40s} {rq:.3f} {rk:.3f} {rv:.3f}")
