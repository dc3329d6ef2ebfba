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
    GPU at all. On a machine with a GPU a missing library is an error, not a
    skip."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_scaled_precision_quantize_gb300 as bsq
    bsq.load()  # raises if the library was not built
    return bsq


# ---------------------------------------------------------------- helpers
def to_dev(a, dtype=None):
    """numpy -> CUDA tensor; uint16 bf16 bit patterns become bf16."""
    import numpy as np
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).cuda()
    t = torch.from_numpy(a).cuda()
    return t if dtype is None else t.to(dtype)


def to_np(t):
    """CUDA tensor -> numpy (bf16 as uint16 bits, fp32 kept)."""
    import numpy as np
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.int16:
        return t.numpy().view(np.uint16)
    return t.numpy()


def bits_equal(a, b):
    """Bitwise equality of two arrays of equal dtype/shape (fp32 compared as
    bit patterns, so -0.0 != 0.0 and NaN payloads matter)."""
    import numpy as np
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    if a.shape != b.shape or a.dtype.itemsize != b.dtype.itemsize:
        return False
    u = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}[a.dtype.itemsize]
    return np.array_equal(a.view(u), b.view(u))


def first_mismatch(a, b):
    import numpy as np
    a = np.asarray(a)
    b = np.asarray(b)
    idx = np.argwhere(a != b)
    if idx.size == 0:
        return None
    i = tuple(idx[0])
    return f"{idx.shape[0]} mismatches; first at {i}: got {a[i]} expected {b[i]}"
