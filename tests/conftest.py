import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads (GPU box only)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library, loaded through the Python binding (GPU tests)."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test collected without a CUDA device")
    import gemm_rtn_sym_gb300 as w4

    w4.load()
    return w4
