import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU case")


@pytest.fixture(autouse=True)
def _support_order(monkeypatch):
    """Contexts built by the tests process attributes in ascending-support order (option value 2),
    so that their closure counts can be compared with the oracle's over the same order; the tests
    of the other values set FCA_ATTR_ORDER themselves."""
    monkeypatch.setenv("FCA_ATTR_ORDER", "2")
