import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def lib():
    """The built CUDA library, loaded; skips nothing -- a GPU test must have it."""
    import torch
    from exact_attention_blackwell_tma_gb300 import binding
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return binding.load()
