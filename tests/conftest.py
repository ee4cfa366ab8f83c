import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libpkv.so")


@pytest.fixture(scope="session")
def cuda():
    """Fails (does not skip) when no GPU is visible: a gpu-marked test must run on the GPU."""
    import torch
    assert torch.cuda.is_available(), "gpu-marked test needs a CUDA device"
    return torch.device("cuda:0")


@pytest.fixture(scope="session")
def built():
    """Builds libpkv.so / libpkv_synth.so in-tree if they are missing or stale (nvcc cross-compiles)."""
    from continuous_batching_paged_ragged_gb300 import _build
    _build.build()
    from continuous_batching_paged_ragged_gb300 import pkv
    return pkv.load()
