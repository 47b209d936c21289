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


@pytest.fixture(autouse=True)
def _no_failed_index_check(request):
    """When the library under test is the debug build (SDPA08_LIBRARY names
    it), every GPU test must end without a failed in-kernel index check."""
    yield
    if not os.environ.get("SDPA08_LIBRARY") or request.node.get_closest_marker("gpu") is None:
        return
    import scaled_dot_product_08_gb300 as sdpa
    st = sdpa.load().attn_get_device_status(None)
    if st == sdpa.Status.CHECK:
        _, info = sdpa.attn_get_timeout_info(None)
        pytest.fail(f"in-kernel index check failed: site {info[0] >> 16:#x}, CTA {info[1]}, thread {info[2]}, "
                    f"index {info[3]}")
