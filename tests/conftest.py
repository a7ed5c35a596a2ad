import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


@pytest.fixture(scope="session")
def lib():
    """The CUDA library's Python binding (built in-tree by __graft_entry__.build)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mxfp8_block_scaled_x4_gb300 as mx
    return mx
