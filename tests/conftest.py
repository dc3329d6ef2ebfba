import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.fixture(scope="session")
def O():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def gpu():
    """The CUDA library on a GPU; the test is skipped only when there is no
    GPU at all. On a GPU machine a missing library is an error, not a skip."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_scaled_precision_quantize_gb300 as bsq
    bsq.load()  # raises if the library was not built
    return bsq
