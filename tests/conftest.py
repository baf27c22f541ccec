import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libcsa2.so")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle


@pytest.fixture(scope="session")
def csa2():
    from fp4_compressed_sparse_csa2_gb300 import build
    build.build()
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from fp4_compressed_sparse_csa2_gb300 import csa2 as lib
    return lib
