import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a B300 (sm_103a) GPU")
    config.addinivalue_line("markers", "slow: long CPU test")


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library, loaded through the package binding."""
    from bounded_kv_cache_la_b300 import capi
    return capi.load()
