import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU")


@pytest.fixture(scope="session")
def smla_lib():
    """libsmla.so, built in-tree if it is missing or stale."""
    from sparse_mla_decode_04_gb300 import _build, smla

    _build.build()
    return smla.load_library()


@pytest.fixture(scope="session")
def cuda_device(smla_lib):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)
