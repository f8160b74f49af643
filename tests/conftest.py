import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda():
    """The CUDA device, or skip when the test runs on a machine without one."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(scope="session")
def hyq(cuda):
    """The loaded CUDA library binding (fails loudly if it cannot be loaded)."""
    import hybrid_precision_quantized_gb300 as hyq
    hyq.load()
    return hyq
