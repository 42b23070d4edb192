import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes on the host side)")


# ROPE_GB300_DEBUG_BOUNDS=1: the GPU tests run on the bounds-checking debug
# build, and after every GPU test the device error word must not report an
# access outside a tensor.
DEBUG_BOUNDS = os.environ.get("ROPE_GB300_DEBUG_BOUNDS", "0") not in ("", "0")


@pytest.fixture(scope="session")
def rope_gpu():
    """The built CUDA library on a GPU machine; skips on a machine without CUDA."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_rope_positional_gb300 import build as B
    import transformer_rope_positional_gb300 as R

    B.build(debug=DEBUG_BOUNDS)
    R.load()
    return R


@pytest.fixture(autouse=True)
def _no_access_outside_a_tensor(request):
    yield
    if not DEBUG_BOUNDS or request.node.get_closest_marker("gpu") is None:
        return
    import torch

    if not torch.cuda.is_available():
        return
    import transformer_rope_positional_gb300 as R

    code = R.get_device_error()
    assert not code & R.ROPE_DEVICE_INDEX_OUT_OF_BOUNDS, "a kernel addressed memory outside a tensor"
