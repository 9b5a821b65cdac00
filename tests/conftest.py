import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")


@pytest.fixture(scope="session")
def sage():
    """The CUDA binding with the in-tree library built (GPU tests only)."""
    import torch
    from int8_quantized_attention_gb300 import binding, build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.lib()
    return binding
