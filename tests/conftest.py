import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built libptb.so")
    config.addinivalue_line(
        "markers", "slow: full-size parity case (minutes of oracle time)")


@pytest.fixture(scope="session")
def ptb_lib():
    """The CUDA path through its Python binding; fails loudly if unbuilt."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test collected without a CUDA device")
    import block_sliding_window_gb300 as bsw
    bsw.load()
    return bsw
