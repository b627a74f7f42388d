import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libfp4idx.so")
    config.addinivalue_line("markers", "slow: long-running CPU test")
    config.addinivalue_line("markers", "fake_ptr: passes fake device pointers that host checks must reject")
    config.addinivalue_line(
        "markers",
        "floor_reading: some compared bytes (all-zero or subnormal groups) are decided by the "
        "scale-floor reading, a value the pages do not print; tests/test_oracle_floors.py shows "
        "which floors give the same bytes")


def pytest_collection_modifyitems(config, items):
    # GPU tests need a device; on a CPU-only machine they are skipped, never
    # silently run on a fallback.
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)
