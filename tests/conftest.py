import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size case")


LAST_MODULES = ("test_zz_no_alloc",)  # run after every other test (see that module's docstring)


def pytest_collection_modifyitems(config, items):
    # the allocation-free entry point's tests go last whatever the file order: if one of them fails, a run that
    # stops at the first failure has already run every other test
    items.sort(key=lambda it: getattr(it.module, "__name__", "").rsplit(".", 1)[-1] in LAST_MODULES)
    # GPU tests cannot run without a device; skip them cleanly when asked for them anyway
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)
