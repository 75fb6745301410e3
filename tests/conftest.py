import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, TESTS):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library (built in-tree on first use)."""
    from dynamic_sparse_attention_indexer_gb300 import _build
    _build.ensure_built()
    from dynamic_sparse_attention_indexer_gb300 import _abi
    return _abi.load()
