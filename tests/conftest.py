import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library binding; a GPU test fails loudly when the library is missing."""
    import engram_conditional_memory_gb300 as ecm
    from engram_conditional_memory_gb300 import build

    build.build()  # no-op when the in-tree library is up to date
    ecm.load_library()
    return ecm
