import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libdsa")
    config.addinivalue_line("markers", "slow: full-size workload")


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library, built in-tree if it is missing."""
    import dsa_sparse_mla_paged_gb300 as dsa

    if not os.path.exists(dsa.library_path()):
        from dsa_sparse_mla_paged_gb300 import _build

        _build.build()
    return dsa.load()


@pytest.fixture(scope="session")
def cuda_ok():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return True
