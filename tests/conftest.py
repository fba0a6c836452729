import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a)")


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library (compiled on first use)."""
    from zero_sharded_optimizer_shard_gb300 import build, zero3
    build.build_all(quiet=True)
    return zero3.load()
