import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The errors every parity check reached (worst per test), so that a quiet run still
    shows how far the CUDA path is from the oracle and from the tolerance."""
    try:
        import parity
    except Exception:
        return
    if not parity.RECORD:
        return
    terminalreporter.write_sep("-", "parity: achieved errors (worst per test)")
    for line in parity.summary_lines():
        terminalreporter.write_line(line)


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle
