import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built libadaln.so")


@pytest.fixture(scope="session")
def oracle():
    """The CPU oracle package (built on first use)."""
    import oracle as o
    o.load()
    return o


def have_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def adaln():
    """The ctypes binding of libadaln.so; GPU tests fail loudly without it."""
    if not have_gpu():
        pytest.fail("GPU test collected on a machine without a CUDA device")
    from adaln_video_dit_gb300 import _lib
    return _lib
