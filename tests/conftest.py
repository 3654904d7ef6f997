import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (GB300, sm_103a); runs the CUDA path")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.Oracle()


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, loaded through its Python binding. GPU tests only."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device in this process")
    import online_softmax_02_gb300 as attn
    attn.load()          # raises loudly if libattn.so is missing
    return attn
