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
    """The fp64 oracle, built on first use."""
    import oracle
    oracle.lib()
    return oracle


@pytest.fixture(scope="session")
def gdn():
    """The CUDA library through its Python binding (built on first use)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_decode_gb300 as g
    g.load()
    return g
