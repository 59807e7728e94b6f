import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libattn")
    config.addinivalue_line("markers", "slow: large parity cases")


def pytest_collection_modifyitems(config, items):
    """The guard-canary tests run after every parity test."""
    items.sort(key=lambda it: os.path.basename(str(it.fspath)) == "test_gpu_canaries.py")


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library through its Python binding (built on demand)."""
    from exact_attention_73_gb300 import binding
    return binding.load(build_if_missing=True)
