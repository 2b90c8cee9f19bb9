import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads")


@pytest.fixture(scope="session")
def lib():
    """The compiled libpagedattn, built in-tree if missing."""
    from paged_kv_decode_24_gb300 import build as _build
    _build.ensure_built()
    from paged_kv_decode_24_gb300 import binding
    return binding.load()
