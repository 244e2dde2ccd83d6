import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built libkda.so")


@pytest.fixture(scope="session")
def kda_lib():
    """Build (if stale) and load the CUDA library; GPU tests depend on it."""
    from kimi_delta_attention_08_gb300 import build, _lib
    build.build()
    return _lib.load()
