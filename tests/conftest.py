import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: longer CPU test")


def pytest_sessionfinish(session, exitstatus):
    from tests._parity import MARGINS
    MARGINS.dump()


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")
