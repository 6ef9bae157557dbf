import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libdn.so")
    config.addinivalue_line("markers", "slow: large CPU-side oracle runs")


@pytest.fixture(scope="session")
def cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a gpu-marked test ran without a CUDA device")
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter):
    # both error measures of every GPU-vs-oracle check, worst case per check name
    from tests import parity
    if not parity.REPORT:
        return
    worst = {}
    for name, e, ee, tol in parity.REPORT:
        w = worst.setdefault((name, tol), [0.0, 0.0, 0])
        w[0], w[1], w[2] = max(w[0], e), max(w[1], ee), w[2] + 1
    terminalreporter.section("parity: per-tensor max|d|/max|ref| (asserted) and element-wise max |d|/(|ref|+1e-3)")
    for (name, tol) in sorted(worst):
        e, ee, n = worst[(name, tol)]
        terminalreporter.write_line("%-28s bar %.0e  checks %4d  per-tensor %.3g  element-wise %.3g" % (
            name, tol, n, e, ee))
