import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def lib():
    """The product binding with its shared library loaded (fails loudly if not built)."""
    import tiled_distributed_attention_gb300 as m
    if not os.path.exists(m.LIB_PATH):
        from tiled_distributed_attention_gb300 import _build
        _build.build()
    m.load_library()
    return m
