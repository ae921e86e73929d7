import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: longer CPU statistical test")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library through its Python binding; GPU tests only."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test collected without a CUDA device")
    import speculative_decoding_verify_08_gb300 as sv
    sv.load()
    return sv
