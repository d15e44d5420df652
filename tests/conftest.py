import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built librr.so")


@pytest.fixture(autouse=True)
def _guard_bands():
    """After every test, the guard bands around each device buffer the parity
    helpers made must still hold their sentinel (no out-of-bounds writes)."""
    yield
    parity = sys.modules.get("parity")
    if parity is not None and parity._GUARDED:
        parity.check_guards(clear=True)
