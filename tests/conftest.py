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
def cuda_dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _guard_bands(request):
    """GPU tests: the guard bands around every array made through tests/_support
    must be intact when the test ends."""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    import _support
    _support.guards_reset()
    yield
    _support.assert_guards_intact()
    _support.guards_reset()
