import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


import pytest


@pytest.fixture(scope="session")
def fa():
    """The CUDA library, built in-tree, on a machine with a GPU."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from exact_io_aware_11_gb300 import build
    build.build()
    import exact_io_aware_11_gb300 as pkg
    pkg.lib()
    return pkg
