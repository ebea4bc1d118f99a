import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def lib():
    """The CUDA library, built in-tree if it is missing."""
    from hybrid_model_ssm_mamba_gb300 import replay
    return replay.load_library(build_if_missing=True)


# One-line measurement summaries the GPU tests report (drift tables and the like); they are
# printed at the end of the run, where the tail of a quiet run's log keeps them.
_REPORTS = []


@pytest.fixture(scope="session")
def report():
    return _REPORTS.append


def pytest_terminal_summary(terminalreporter):
    if _REPORTS:
        terminalreporter.section("measurements reported by the tests")
        for line in _REPORTS:
            terminalreporter.write_line(line)
