import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes of oracle time)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The loaded C-ABI library on a GPU machine (gpu tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test collected on a machine without a CUDA device")
    import scaled_dot_product_08_gb300 as sdpa
    sdpa.load()
    return sdpa
