import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (runs the CUDA library)")
    config.addinivalue_line("markers", "slow: a longer CPU test")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()
