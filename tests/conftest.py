import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library on a GPU machine. The CUDA path has no CPU
    fallback: a missing GPU skips these tests, and a missing library fails."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hybrid_ssm_decode_gb300 as rssm
    rssm.load()  # raises if the library is missing or stale
    return rssm
