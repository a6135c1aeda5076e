import os
import sys

import pytest

_TESTS = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_TESTS)
for p in (_ROOT, _TESTS):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); run with -m gpu")


@pytest.fixture(scope="session")
def gemv_lib():
    """The compiled C-ABI library (built in-tree on first use)."""
    from memory_bound_gemv_02_gb300 import _build
    _build.ensure_built()
    import memory_bound_gemv_02_gb300 as g
    return g


@pytest.fixture(scope="session")
def cuda_dev(gemv_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected but no CUDA device is visible")
    torch.cuda.init()
    return torch.device("cuda", torch.cuda.current_device())
