import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload, minutes of host work")


def _have_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    """Skip GPU tests without a device, unless PGQA_REQUIRE_GPU=1 (then they fail)."""
    if _have_gpu() or os.environ.get("PGQA_REQUIRE_GPU") == "1":
        return
    skip = pytest.mark.skip(reason="no CUDA device (set PGQA_REQUIRE_GPU=1 to fail instead)")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
