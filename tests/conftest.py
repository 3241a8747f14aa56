import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity cases (minutes)")


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library through its Python binding (built by __graft_entry__.build())."""
    from transformer_sharding_affinity_gb300 import binding
    return binding.load()
