import sys
from pathlib import Path

import pytest

REPO = Path(__file__).resolve().parent.parent
if str(REPO) not in sys.path:
    sys.path.insert(0, str(REPO))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and libfd.so")
    config.addinivalue_line("markers", "slow: takes more than a few seconds of CPU time")


@pytest.fixture(scope="session")
def fdlib():
    """Build libfd.so if stale and load it (the library loads without a GPU)."""
    from memory_bound_decode_fd_gb300 import build

    build.build()
    import memory_bound_decode_fd_gb300 as fd

    return fd.load_library()


@pytest.fixture(scope="session")
def cuda_device(fdlib):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")
