import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libswa.so")
    config.addinivalue_line("markers", "slow: long-running GPU case (full-size workloads)")


@pytest.fixture(scope="session")
def cuda_device():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(scope="session")
def swa(cuda_device):
    """The CUDA library binding; fails loudly (no fallback) when the extension is missing."""
    import sliding_window_flash_gb300 as swa_mod

    swa_mod.load()  # raises if libswa.so is absent
    return swa_mod
