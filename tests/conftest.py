import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a library)")
    config.addinivalue_line("markers", "slow: long-running test")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def qw():
    """The CUDA library's Python binding, built in-tree if needed (GPU tests only)."""
    if not gpu_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    import decode_qwen3_decoder_gb300 as pkg
    pkg.build()
    return pkg
