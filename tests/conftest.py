import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built CUDA library")


@pytest.fixture(scope="session", autouse=True)
def _native_libraries():
    """The CUDA library, the input generator and the oracle are built once per
    session if missing or stale (nvcc cross-compiles without a GPU)."""
    import __graft_entry__
    __graft_entry__.build()
