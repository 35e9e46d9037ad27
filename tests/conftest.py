import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library)")
    config.addinivalue_line("markers", "slow: large CPU case")


def pytest_collection_modifyitems(config, items):
    # A test file whose name starts with test_zz_ runs after every other file.
    items.sort(key=lambda it: os.path.basename(str(it.fspath)).startswith("test_zz_"))


@pytest.fixture(scope="session")
def ep():
    """The CUDA library's Python binding, built in-tree if needed."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_get_dispatch_04_gb300 import build as ep_build
    ep_build.build()
    import combine_get_dispatch_04_gb300 as ep_mod
    ep_mod.load()
    return ep_mod
