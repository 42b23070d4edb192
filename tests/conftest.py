import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes on the host side)")


@pytest.fixture(scope="session")
def rope_gpu():
    """The built CUDA library on a GPU machine; skips on a machine without CUDA."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_rope_positional_gb300 import build as B
    import transformer_rope_positional_gb300 as R

    B.build()
    R.load()
    return R
