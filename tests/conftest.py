import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def built_lib():
    """Path of liblinattn.so, building it (nvcc cross-compile, no GPU needed) if stale."""
    from linear_attention_chunked_conv1d_gb300 import build
    return build.build()


@pytest.fixture(scope="session")
def cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_chunked_conv1d_gb300 import build
    build.build()
    return torch.device("cuda:0")
