import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libgdn.so")


@pytest.fixture(scope="session")
def gdn():
    """The ctypes binding to libgdn.so (built in-tree if needed)."""
    from gated_deltanet_chunked_gb300 import gdn as binding

    binding.load()
    return binding


@pytest.fixture(scope="session")
def cuda():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")
