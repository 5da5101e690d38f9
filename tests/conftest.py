import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a); calls the kernels through the C ABI")


@pytest.fixture(scope="session")
def cuda():
    """The CUDA device; a GPU test fails (it does not skip) when there is none,
    so a missing GPU or a missing library can never pass silently."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("this test needs a CUDA GPU")
    import invariant_bi_rmsnorm_02_gb300 as bi
    bi.load()  # raises if the CUDA library is missing
    return torch.device("cuda", 0)
