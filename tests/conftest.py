import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, built in-tree if needed; its calls need a GPU."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_151_gb300 import pa
    pa.load()
    return pa
