import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300) and the built CUDA library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.lib()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """Selection ties of the GPU parity tests: heads whose page set differs from
    the oracle's only by pages whose fp64 score is within the tie window of the
    decision boundary."""
    try:
        from gpu_util import TIES
    except Exception:
        return
    if not TIES:
        return
    heads = sum(n for _, n, _ in TIES)
    ties = sum(t for _, _, t in TIES)
    terminalreporter.write_line(
        f"selection ties: {ties} of {heads} compared heads differ from the oracle only at the "
        f"decision boundary ({sum(1 for _, _, t in TIES if t)} of {len(TIES)} comparisons)")
