import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large CPU oracle work")


@pytest.fixture(scope="session")
def msa():
    """The product binding (C-ABI library loaded through ctypes)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_block_sparse_gb300 as m
    m.load()           # raises if the shared library is missing: no fallback
    return m
