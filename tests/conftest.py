import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the compiled CUDA library")


@pytest.fixture(scope="session")
def lib():
    """The compiled C-ABI library (GPU tests only)."""
    import mla_latent_kv_09_gb300 as m
    return m
