import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")

import pytest


@pytest.fixture(scope="session")
def granikv_lib():
    """Build libgranikv.so in-tree if it is missing or stale, then load it."""
    from shared_prefix_kv_decode_gb300 import build as _build
    from shared_prefix_kv_decode_gb300 import _binding
    _build.build()
    return _binding.load_library()


@pytest.fixture(scope="session")
def cuda_ok(granikv_lib):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return True
