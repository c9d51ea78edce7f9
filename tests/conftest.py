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
    config.addinivalue_line("markers", "gpu: needs a CUDA device (runs the CUDA library)")
    config.addinivalue_line("markers", "slow: a longer CPU test")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()


@pytest.fixture(scope="session")
def linattn():
    """The CUDA library's Python binding, built in-tree first if needed."""
    from kernelized_causal_attention_gb300 import _build
    _build.build()
    import kernelized_causal_attention_gb300 as la
    la.lib()
    return la


@pytest.fixture(scope="session")
def cuda(linattn):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter):
    """Per test: the largest normwise error (asserted) and the largest
    elementwise relative error (reported only) of its GPU results."""
    from errstats import RECORDS
    if not RECORDS:
        return
    worst = {}
    for test, norm, elem in RECORDS:
        n, e = worst.get(test, (0.0, 0.0))
        worst[test] = (max(n, norm), max(e, elem))
    terminalreporter.section("GPU vs oracle: normwise max / elementwise relative (reported)")
    for test, (n, e) in sorted(worst.items()):
        terminalreporter.write_line(f"{n:10.3e} {e:10.3e}  {test}")
