import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built library")


def pytest_collection_modifyitems(config, items):
    # Keep tests that need a GPU from erroring out on a CPU-only machine when
    # they are selected explicitly: skip them with a clear reason instead.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU on this machine")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    # The parity figures of every check, for a table of measured errors.
    path = os.environ.get("FA_PARITY_REPORT")
    if not path:
        return
    try:
        from tests import parity
    except Exception:  # the GPU helpers were never imported
        return
    import json
    with open(path, "w") as f:
        json.dump(parity.REPORTS, f, indent=1)
