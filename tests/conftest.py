import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the kernels through the C ABI)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library, on a machine with a CUDA device."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from first_order_linear_gb300 import _lib, build
    build.build()
    return _lib.load()
