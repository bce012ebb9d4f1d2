import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def gdnlib():
    """The CUDA library, built in-tree if needed; GPU tests fail loudly without it."""
    import torch
    from linear_attention_decode_gb300 import binding, build
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    build.build()
    return binding.load_library()
