import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libtgc.so")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session", autouse=True)
def _library_built():
    """libtgc.so is compiled in-tree (nvcc for sm_103a) if it is missing or older than its sources."""
    from tile_gather_comm_gb300 import _build
    _build.build()
