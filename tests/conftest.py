import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if gpu_available():
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    """Write every parity comparison of the session to $LAT_PARITY_REPORT (if set)."""
    path = os.environ.get("LAT_PARITY_REPORT")
    if not path:
        return
    try:
        from tests.parity import REPORT
    except Exception:
        return
    with open(path, "w") as f:
        for what, val, bound in REPORT:
            f.write(f"{what}\t{val:.4e}\t{bound:.1e}\n")
