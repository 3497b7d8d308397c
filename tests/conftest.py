import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes of host work)")


@pytest.fixture(scope="session")
def cuda():
    """The CUDA device for parity tests; these tests need a GPU and the native library."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rope_tfk_rmsnorm_gb300 as tfk
    tfk.load()  # raises if libtfk.so is missing or does not load
    return torch.device("cuda", 0)
