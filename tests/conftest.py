import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running (large host-memory stacks)")


def pytest_collection_modifyitems(config, items):
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(autouse=True)
def _cuda_state_is_clean(request):
    """Every GPU test starts and ends with a usable CUDA state (a pending error
    left by one test must not be charged to the next)."""
    if "gpu" not in request.keywords:
        yield
        return
    import torch
    torch.ones(1, device="cuda").add_(1)
    torch.cuda.synchronize()
    yield
    torch.ones(1, device="cuda").add_(1)
    torch.cuda.synchronize()
