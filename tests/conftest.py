import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle._default()


@pytest.fixture(scope="session")
def lib():
    """The CUDA library, built in-tree if it is missing (nvcc cross-compiles
    without a GPU)."""
    from paged_kv_decode_fa_gb300 import build as b
    b.build()
    import paged_kv_decode_fa_gb300 as fa
    return fa


@pytest.fixture(scope="session")
def cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_fa_gb300 import build as b
    b.build()
    return torch.device("cuda:0")
