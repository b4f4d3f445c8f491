import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running (large shapes)")


@pytest.fixture(scope="session")
def dtp():
    """The C-ABI library through its Python binding (built in-tree on first use)."""
    import dense_transformer_prefill_gb300 as pkg
    pkg.build()
    return pkg
