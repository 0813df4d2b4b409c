import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built libh3attn")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def h3():
    """The CUDA library binding; GPU tests fail loudly if it cannot load."""
    if not gpu_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    import video_dit_dense_gb300 as h3
    h3.load()
    return h3
