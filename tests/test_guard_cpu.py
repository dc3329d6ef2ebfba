"""The guard-band helper the GPU tests rely on, exercised on CPU tensors: a
write one element past an output, or one before it, is reported; writes
inside it are not."""
import pytest
import torch

from conftest import GuardedBuffer, _GuardedTorch, guarded_empty


def test_guard_accepts_writes_inside():
    buf, t = guarded_empty((7, 5), torch.float32, device="cpu")
    t.fill_(1.0)
    buf.check()


@pytest.mark.parametrize("where", ["before", "after"])
def test_guard_reports_a_write_outside(where):
    buf, t = guarded_empty((3, 16), torch.uint8, device="cpu")
    t.fill_(0)
    # the planted mistake: one byte just outside the output
    off = 4095 if where == "before" else 4096 + t.numel()
    buf.raw[off] = 0
    with pytest.raises(AssertionError, match="write outside"):
        buf.check()


def test_guarded_torch_carves_cuda_allocations_only():
    reg = []
    g = _GuardedTorch(torch, reg)
    c = g.empty(4, 4, dtype=torch.float32, device="cpu")
    assert c.shape == (4, 4) and not reg
    assert g.float32 is torch.float32
    buf = GuardedBuffer(0, "cpu")
    assert buf.view((0, 256), torch.bfloat16).shape == (0, 256)
    buf.check()
