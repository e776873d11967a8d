import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload, minutes")


def _cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def kvp():
    """The package, built for sm_103a; GPU tests only."""
    if not _cuda_ok():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import kv_cache_pruning_gb300 as pkg
    return pkg
