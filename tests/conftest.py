import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def ekv_lib():
    """The ekv C-ABI binding; builds the shared library first when it is missing."""
    from mixed_precision_paged_gb300 import build
    build.ensure_built()
    from mixed_precision_paged_gb300 import ekv
    return ekv
