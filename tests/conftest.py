import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libkvc.so")
    config.addinivalue_line("markers", "slow: long-running parity case")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def kvc_lib():
    """Builds libkvc.so in-tree if needed (nvcc cross-compiles without a GPU) and loads it."""
    from kv_cache_append_rope_gb300 import build
    build.build()
    from kv_cache_append_rope_gb300 import _lib
    return _lib
