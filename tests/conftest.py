import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a); calls the CUDA library "
        "through its C ABI")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    """With DSA_PARITY_REPORT=<file>, write every output comparison of the
    run (test, tensor, max error, max |oracle|, their ratio) as JSON lines:
    the measured normalised errors of the parity checks."""
    path = os.environ.get("DSA_PARITY_REPORT")
    if not path:
        return
    import json
    from tests.helpers import PARITY_LOG
    with open(path, "w") as f:
        for test, name, err, top in PARITY_LOG:
            f.write(json.dumps({"test": test, "tensor": name, "max_err": err,
                                "max_ref": top,
                                "ratio": err / top if top else None}) + "\n")
