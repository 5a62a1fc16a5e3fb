import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("this test is marked gpu but no CUDA device is visible")
    return torch.device("cuda", 0)


@pytest.fixture(params=["flat", "ring"])
def swiglu_kernel(request, monkeypatch):
    """The library has two bit-identical kernels for the SwiGLU forward cast,
    a flat stream and a TMA ring, and picks one by a measured rule (weight,
    input size); a test that takes this fixture runs once through each."""
    monkeypatch.setenv("TKQ_SWIGLU_KERNEL", request.param)
    return request.param
