import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads")


@pytest.fixture(scope="session")
def lynx():
    """The CUDA library binding, built in-tree; GPU tests fail (not skip) if it is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected without a visible CUDA device")
    import activation_sparse_linear_gb300 as asl
    return asl
