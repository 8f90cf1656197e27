import os
import sys

import pytest

TESTS = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(TESTS)
for p in (ROOT, TESTS):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the libkvo kernels)")


@pytest.fixture(scope="session")
def kvo_lib():
    """The built libkvo (built in-tree on first use)."""
    from host_ram_tiered_gb300 import build, kvo
    build.build()
    return kvo.load()
