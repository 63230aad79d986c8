import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


def _cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _cuda_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """The largest error relative to (|A||B|)_ij of every full-size parity
    comparison that ran, per problem and mode."""
    rows = sys.modules.get("tests._gpu")
    rows = getattr(rows, "ERROR_REPORT", None) if rows else None
    if not rows:
        return
    terminalreporter.section("max |C - C_oracle| / (|A||B|)_ij over every element")
    for what, ratio, tol in rows:
        terminalreporter.write_line("%-34s %.3e  (bound %.0e)" % (what, ratio, tol))
