import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); run with -m gpu")
    config.addinivalue_line("markers", "slow: full-size workloads")


@pytest.fixture(scope="session")
def splitzip_lib():
    """The C-ABI library, built in-tree if it is missing or stale."""
    from lossless_kv_cache_gb300 import build_lib
    import lossless_kv_cache_gb300 as sz

    build_lib.build()
    return sz.lib()
