import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libattn")
    config.addinivalue_line("markers", "slow: large parity cases")


LAST = ("test_gpu_bench_config.py", "test_gpu_canaries.py", "test_zz_no_alloc.py")


def pytest_collection_modifyitems(config, items):
    """The benchmark-configuration, guard-canary and allocation-free backward
    tests run after every other test, in that order."""
    def rank(item):
        name = os.path.basename(str(item.fspath))
        return LAST.index(name) + 1 if name in LAST else 0
    items.sort(key=rank)


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library through its Python binding (built on demand)."""
    from exact_attention_73_gb300 import binding
    return binding.load(build_if_missing=True)
