import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload")


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA binding, built in-tree if needed; skip-free: a GPU test that
    cannot load the library fails."""
    import torch
    assert torch.cuda.is_available(), "gpu tests need a CUDA device"
    import moe_grouped_gemm_device_gb300 as rg
    rg.load()
    return rg
