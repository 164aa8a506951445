import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103)")
    config.addinivalue_line("markers", "slow: long-running oracle comparison")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def lib():
    """The compiled C-ABI library (built in-tree on first use)."""
    from block_diffusion_drafter_gb300 import _build
    _build.build_library()
    import block_diffusion_drafter_gb300 as dfl
    return dfl
