import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running case")


@pytest.fixture(scope="session")
def gdn():
    """The CUDA binding; GPU tests fail loudly if the library or the GPU is missing."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test collected without a CUDA device")
    from gated_deltanet_cpr_gb300 import api

    api.load()  # raises if the shared library is missing
    return api
