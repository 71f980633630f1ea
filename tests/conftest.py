import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads (seconds to minutes)")


def pytest_collection_modifyitems(config, items):
    """GPU tests fail loudly (not skip) when no GPU is visible: a silent skip
    on a GPU machine would hide a broken path."""
    return
