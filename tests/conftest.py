import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

_PARITY = pytest.StashKey[list]()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")
    config.stash[_PARITY] = []


@pytest.fixture
def parity_log(request):
    """log(name, err, tol): records a parity result for the end-of-run summary."""
    def log(name, err, tol):
        request.config.stash[_PARITY].append((name, float(err), float(tol)))
    return log


def pytest_terminal_summary(terminalreporter):
    rows = terminalreporter.config.stash.get(_PARITY, [])
    if not rows:
        return
    terminalreporter.write_line("parity against the oracle, every element "
                                "(max|gpu - oracle| / max|oracle|, tolerance):")
    for name, err, tol in rows:
        terminalreporter.write_line(f"  {name}: {err:.3g} (tol {tol:g})")
