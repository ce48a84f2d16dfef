import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")


@pytest.fixture
def rng():
    return np.random.default_rng(12345)


def _cuda_available():
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def lib():
    """The compiled C-ABI library (built in-tree on first use)."""
    import __graft_entry__

    __graft_entry__.build()
    import rope_qkv_prologue_gb300 as qp

    return qp


@pytest.fixture(scope="session")
def cuda(lib):
    if not _cuda_available():
        pytest.skip("no CUDA device")
    import torch

    torch.cuda.init()
    return torch.device("cuda:0")
