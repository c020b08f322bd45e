import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """Print the achieved parity errors against their tolerances."""
    try:
        import _margins
    except ImportError:
        return
    if not _margins.RECORDS:
        return
    terminalreporter.write_sep("-", "achieved parity errors (error / tolerance)")
    for name, err, tol in _margins.RECORDS:
        terminalreporter.write_line(f"{err:10.3e} / {tol:8.1e}  ({err / tol:6.3f})  {name}")
