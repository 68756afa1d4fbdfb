import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (run with -m gpu)")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library binding, built if needed.  GPU tests only."""
    if not gpu_available():
        pytest.fail("test marked gpu but no CUDA device is visible")
    import quantized_kv_decode_paged_gb300 as qk
    qk.load_library()
    return qk
