import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads (several GB of device memory)")


@pytest.fixture(scope="session")
def lib():
    """The product library (C ABI through the Python binding); GPU tests only."""
    import kv_cache_eviction_tria_gb300 as tria
    tria.load_library()
    return tria
