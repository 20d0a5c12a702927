import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built CUDA library")


@pytest.fixture(scope="session", autouse=True)
def _host_libraries():
    """The oracle (gcc) and the input generator (nvcc, host + device code) are
    built once per session if missing or stale."""
    from oracle import _build as oracle_build
    from workloads import _build as synth_build
    oracle_build.build()
    synth_build.build()
