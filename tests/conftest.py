import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")


def pytest_collection_modifyitems(config, items):
    # GPU tests need a device: skip them cleanly when none is present so that
    # `-m "not gpu"` and plain runs on a CPU host stay green.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    # every GPU-vs-oracle comparison's metrics (normwise error and bound,
    # elementwise excesses against the exact-accumulation and the sequential
    # oracle results), one JSON line each, when EMU_PARITY_REPORT names a file
    path = os.environ.get("EMU_PARITY_REPORT")
    if not path:
        return
    try:
        from tests import _gpu
    except Exception:
        return
    import json
    with open(path, "a") as f:
        for r in _gpu.REPORT:
            f.write(json.dumps(r) + "\n")
