import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libbeamdec")
    config.addinivalue_line("markers", "slow: long CPU case")


@pytest.fixture(scope="session")
def gpu_lib():
    """The loaded CUDA library; GPU tests fail (not skip) when it is missing."""
    import torch
    assert torch.cuda.is_available(), "GPU test run without a visible CUDA device"
    from wide_beam_generative_gb300 import beamdec
    return beamdec.lib()
