import os
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built libfa2.so")


@pytest.fixture(scope="session")
def fa2_lib():
    """The CUDA library, built in-tree if it is missing or stale."""
    from exact_attention_64_gb300 import build

    build.build()
    import exact_attention_64_gb300 as fa2

    fa2.load_library()
    return fa2


@pytest.fixture(scope="session")
def cuda_device(fa2_lib):
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    return torch.device("cuda:0")
