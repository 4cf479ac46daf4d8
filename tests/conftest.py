import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and libattnres.so")


def cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def gpu():
    """Skip when no GPU is visible; on a GPU machine the CUDA library must load."""
    if not cuda_available():
        pytest.skip("no CUDA device")
    from transformer_depth_wise_gb300 import _lib
    _lib.lib()  # raises if libattnres.so is missing: no fallback path exists
    import torch
    return torch.device("cuda:0")
