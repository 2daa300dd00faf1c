import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the sm_103a library")
    config.addinivalue_line("markers", "slow: longer CPU or GPU cases")


@pytest.fixture(scope="session")
def product_lib():
    """libmamba2.so, built in-tree with nvcc if it is missing or stale."""
    from selective_scan_gb300 import build as b
    b.build()
    import selective_scan_gb300 as ss
    return ss.library()
