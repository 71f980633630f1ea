import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _ensure_library():
    """Build libh3kv.so in-tree if it is missing (nvcc compiles it for sm_103a
    with or without a GPU present), so the binding never silently falls back."""
    lib = os.path.join(ROOT, "store_h3kv_build_gb300", "libh3kv.so")
    if not os.path.exists(lib):
        from store_h3kv_build_gb300 import build_lib
        build_lib.build()


def pytest_configure(config):
    _ensure_library()
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads (seconds to minutes)")


@pytest.fixture(scope="session")
def cuda():
    """GPU tests fail loudly (they never skip) when no sm_103 GPU is visible."""
    import torch
    assert torch.cuda.is_available(), "no CUDA device visible"
    major, minor = torch.cuda.get_device_capability(0)
    assert (major, minor) == (10, 3), f"needs sm_103, found sm_{major}{minor}"
    return torch.device("cuda:0")
