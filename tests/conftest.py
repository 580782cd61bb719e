import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long CPU test")


@pytest.fixture(scope="session")
def bss():
    """The product library, required to be the real CUDA build on a GPU machine."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_sparse_spatio_gb300 as b
    b.load()
    return b
