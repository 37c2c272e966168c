import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    try:
        from gpu_util import ERRORS
    except Exception:
        return
    if ERRORS:
        terminalreporter.write_line("max |out - oracle| per attention test:")
        for k, v in sorted(ERRORS.items()):
            terminalreporter.write_line(f"  {v:.3e}  {k}")
