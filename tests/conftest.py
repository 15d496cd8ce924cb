import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity cases")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """The largest accumulation error the GPU parity checks saw (tests/parity_util.py)."""
    mod = sys.modules.get("parity_util")
    rec = getattr(mod, "RECORD", None)
    if rec:
        terminalreporter.write_line(
            "parity: %d checks, largest accumulation error %.4g x |alpha| sum|a b| (secondary bound %s)"
            % (len(rec), max(rec), mod.SECONDARY_REL))
