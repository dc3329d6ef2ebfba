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


# ---------------------------------------------------------------- guard bands
# compute-sanitizer is not available on the GPU pool, so the GPU tests watch
# for out-of-bounds writes themselves: every output sits inside a larger
# buffer filled with a canary byte, and the bytes before and after it must
# come back unchanged.
CANARY = 0xA5
GUARD_BYTES = 4096


class GuardedBuffer:
    """A device buffer of `nbytes` with GUARD_BYTES of canary on each side;
    the interior starts filled with the canary too (like uninitialised
    memory), so an output element a kernel never writes shows up as a
    mismatch."""

    def __init__(self, nbytes, device):
        import torch
        self.nbytes = int(nbytes)
        self.raw = torch.full((self.nbytes + 2 * GUARD_BYTES,), CANARY, dtype=torch.uint8, device=device)

    def view(self, shape, dtype):
        import torch
        inner = self.raw[GUARD_BYTES:GUARD_BYTES + self.nbytes]
        if dtype != torch.uint8:
            inner = inner.view(dtype)
        return inner.view(tuple(shape))

    def check(self):
        head = self.raw[:GUARD_BYTES]
        tail = self.raw[GUARD_BYTES + self.nbytes:]
        bad_head = int((head != CANARY).sum().item())
        bad_tail = int((tail != CANARY).sum().item())
        assert bad_head == 0 and bad_tail == 0, (
            f"write outside a {self.nbytes}-byte output: {bad_head} guard bytes changed before it, "
            f"{bad_tail} after it")


def guarded_empty(shape, dtype, device="cuda"):
    """(buffer, tensor): an uninitialised-looking tensor inside guard bands;
    call buffer.check() after the kernels that write it have finished."""
    import torch
    shape = tuple(int(s) for s in shape)
    n = 1
    for s in shape:
        n *= s
    itemsize = torch.empty((), dtype=dtype).element_size()
    buf = GuardedBuffer(n * itemsize, device)
    return buf, buf.view(shape, dtype)


class _GuardedTorch:
    """Stands in for the binding module's `torch`: CUDA tensors from
    torch.empty / torch.zeros come from guarded buffers (recorded for the
    check); everything else is torch itself."""

    def __init__(self, real, registry):
        self._real = real
        self._registry = registry

    def __getattr__(self, name):
        return getattr(self._real, name)

    def _is_cuda(self, device):
        return device is not None and self._real.device(device).type == "cuda"

    def empty(self, *size, dtype=None, device=None, **kw):
        if not self._is_cuda(device) or kw:
            return self._real.empty(*size, dtype=dtype, device=device, **kw)
        shape = tuple(size[0]) if len(size) == 1 and isinstance(size[0], (tuple, list)) else size
        buf, t = guarded_empty(shape, dtype or self._real.get_default_dtype(), device)
        self._registry.append(buf)
        return t

    def zeros(self, *size, dtype=None, device=None, **kw):
        if not self._is_cuda(device) or kw:
            return self._real.zeros(*size, dtype=dtype, device=device, **kw)
        t = self.empty(*size, dtype=dtype, device=device)
        t.zero_()
        return t


@pytest.fixture(autouse=True)
def _guard_binding_outputs(request):
    """For every GPU test: each device tensor the binding allocates (outputs,
    workspaces) sits inside canary guard bands, checked after the test."""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    import torch
    if not torch.cuda.is_available():
        yield
        return
    import block_scaled_precision_quantize_gb300 as bsq
    registry = []
    real = bsq.torch
    bsq.torch = _GuardedTorch(real, registry)
    try:
        yield
    finally:
        bsq.torch = real
    torch.cuda.synchronize()
    for buf in registry:
        buf.check()
