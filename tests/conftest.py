import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def nv():
    """The CUDA library (built in-tree if needed). GPU tests fail loudly without it."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_w4a16_moe_gb300 as nvmod
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return nvmod
