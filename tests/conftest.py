import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running case")


def _has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


HAS_GPU = _has_gpu()


def pytest_collection_modifyitems(config, items):
    if HAS_GPU:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def _no_device_error(request):
    """After every GPU test: the library's device error word must be clear
    (a bounded wait inside a kernel that gave up would have set it)."""
    yield
    if not HAS_GPU or "gpu" not in request.keywords:
        return
    import ctypes
    import torch
    from sparse_head_self_gb300 import _native
    torch.cuda.synchronize()
    code = ctypes.c_uint(0)
    _native.check(_native.lib().fibatt_device_error(1, ctypes.byref(code)))
    assert code.value == 0, f"device error word set: {code.value:#x}"
