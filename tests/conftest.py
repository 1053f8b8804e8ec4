import os
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and runs the CUDA library")
    config.addinivalue_line("markers", "slow: long-running")


@pytest.fixture(scope="session")
def profk_lib():
    """The C-ABI library, built in-tree if it is missing or stale (nvcc needed)."""
    from streaming_selection_primitive_gb300.build import build

    build()
    import streaming_selection_primitive_gb300 as pk

    return pk


@pytest.fixture(scope="session")
def cuda_device():
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    return torch.device("cuda:0")


@pytest.fixture()
def pk(profk_lib):
    """The package with options reset to their defaults around each test."""
    profk_lib.reset_options()
    yield profk_lib
    profk_lib.reset_options()
    profk_lib.set_workspace(None)
