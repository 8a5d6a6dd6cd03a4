import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def _cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


@pytest.fixture(scope="session")
def qk():
    """The CUDA library binding; a GPU test fails loudly if it cannot load."""
    if not _cuda_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    from quantised_gguf_weight_gb300 import qk as _qk
    _qk.load()
    return _qk


@pytest.fixture(scope="session")
def orc():
    from oracle import oracle as _o
    _o.build()
    return _o
