"""GPU: the grouped GEMM's bounded waits end in an error status, not a hang.

A test-only copy of the library has its GEMM compiled with a stall hook: the
producer never issues a copy and never arrives, and every wait gives up after
a few thousand polls.  Nothing asynchronous is ever in flight in it, so each
role takes its timeout path safely: the call must return, the status word
must read BSQ_DEV_TIMEOUT, and the CTAs must free their tensor memory -- a
normal GEMM on the same stream right afterwards (which allocates tensor
memory on the same SMs) completes and matches the oracle."""
import ctypes

import numpy as np
import pytest
import torch

from block_scaled_precision_quantize_gb300 import synth
from conftest import to_dev, to_np

pytestmark = pytest.mark.gpu


def _stall_gemm(gpu):
    L = ctypes.CDLL(gpu._build.build_gemm_stall_test_lib())
    fn = L.grouped_expert_gemm_fp4
    fn.restype = ctypes.c_int
    fn.argtypes = gpu._SIGS["grouped_expert_gemm_fp4"][1]
    return fn


def _gemm_case(gpu, M, experts):
    x = synth.normal_with_outliers(M, 256, seed=M)
    w = synth.normal((experts, 128, 256), seed=experts, std=0.02)
    xc, xs, xt = gpu.quantize_nvfp4_per_token(to_dev(x), swizzled=True)
    wc, ws, wt = gpu.quantize_nvfp4_per_expert(to_dev(w), swizzled=True)
    per = M // experts
    offsets = to_dev(np.arange(experts + 1, dtype=np.int32) * per)
    return x, w, (xc, xs, xt, offsets, wc, ws, wt)


@pytest.mark.parametrize("M,experts", [(128, 1), (512, 4)])
def test_gemm_wait_timeout_reports_and_recovers(gpu, O, M, experts):
    stall = _stall_gemm(gpu)
    x, w, (xc, xs, xt, offsets, wc, ws, wt) = _gemm_case(gpu, M, experts)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(M, 128, dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = stall(p(xc), p(xs), p(xt), p(offsets), experts, M, 256, 128, p(wc), p(ws), p(wt), gpu.EPI_F32, p(out), 128,
               gpu.SF_SWIZZLED, p(status), stream)
    assert st == 0, st
    torch.cuda.synchronize()
    assert int(status.item()) == gpu.DEV_TIMEOUT
    assert not out.any()  # the epilogue stored nothing

    # the product GEMM on the same stream: the context is usable and the
    # tensor memory of every SM the stalled CTAs ran on was freed
    status2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = gpu.grouped_expert_gemm_fp4(xc, xs, xt, offsets, wc, ws, wt, dev_status=status2)
    torch.cuda.synchronize()
    assert int(status2.item()) == 0
    oc, osf, ot = O.nvfp4_quantize_rows(x)
    g = to_np(got).astype(np.float64)
    per = M // experts
    for e in range(experts):
        c, s, t = O.nvfp4_quantize_group(w[e:e + 1])
        ref, ab = O.gemm_nvfp4(oc[e * per:(e + 1) * per], osf[e * per:(e + 1) * per], ot[e * per:(e + 1) * per],
                               c[0], s[0], t[0])
        ge = g[e * per:(e + 1) * per]
        assert np.all(np.abs(ge - ref) <= 1e-4 * ab + 1e-30)
        assert np.linalg.norm(ge - ref) <= 1e-5 * np.linalg.norm(ref)
