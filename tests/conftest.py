import multiprocessing as mp
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA path)")


@pytest.fixture(scope="session")
def root():
    return ROOT


@pytest.fixture(scope="session")
def pool():
    """A process pool for the CPU oracle (tests/oracle_pool.py).  Spawned,
    not forked: the test process may already hold a CUDA context."""
    with mp.get_context("spawn").Pool(max(1, min(32, os.cpu_count() or 1))) as p:
        yield p
