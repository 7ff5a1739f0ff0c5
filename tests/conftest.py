import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload")


@pytest.fixture(scope="session", autouse=True)
def _library_built():
    """The C library the tests load, built (or found up to date) once per test
    process before any test runs; parallel workers take turns on the build's
    lock file."""
    from paged_gqa_decode_02_gb300 import build
    build.build()
