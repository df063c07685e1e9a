import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long CPU test")


@pytest.fixture(scope="session", autouse=True)
def _cuda_side_stream():
    """GPU tests run on a created stream (as the benchmark does), so the
    library's programmatic-dependent-launch path is the one exercised."""
    import torch
    if torch.cuda.is_available():
        torch.cuda.set_stream(torch.cuda.Stream())
    yield
