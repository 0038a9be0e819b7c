import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")


@pytest.fixture(scope="session")
def native_lib():
    """The built C-ABI library (built in-tree first if it is missing or stale)."""
    from swiglu_gated_mlp_gb300 import build as _build
    _build.build_library()
    from swiglu_gated_mlp_gb300 import _native
    return _native
