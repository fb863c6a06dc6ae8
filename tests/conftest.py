import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload, minutes on the host side")


@pytest.fixture(scope="session")
def kvc():
    """The CUDA library's Python binding, built in-tree if it is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_kvc_gb300 as k
    if not os.path.exists(k.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    k.load()
    return k
