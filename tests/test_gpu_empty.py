"""GPU: zero-size inputs at every entry point return OK, launch nothing that
touches memory, and leave the device usable: no rows, no tokens, no experts,
or experts that all received zero rows."""
import numpy as np
import pytest
import torch

from block_scaled_precision_quantize_gb300 import synth
from conftest import to_dev

pytestmark = pytest.mark.gpu


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def test_mxfp8_no_rows(gpu):
    x = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    st = _status()
    gpu.quantize_mxfp8_rowcol(x, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_requant_no_rows(gpu):
    codes = torch.empty(0, 128, dtype=torch.uint8, device="cuda")
    sf = torch.empty(0, 16, dtype=torch.uint8, device="cuda")
    scale = torch.empty(0, dtype=torch.float32, device="cuda")
    st = _status()
    gpu.requant_transpose_sr(codes, sf, scale, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_per_expert_no_experts(gpu):
    w = torch.empty(0, 128, 256, dtype=torch.bfloat16, device="cuda")
    gpu.quantize_nvfp4_per_expert(w)
    torch.cuda.synchronize()


def test_gemm_no_rows(gpu):
    E, N, K = 2, 256, 256
    st = _status()
    out = gpu.grouped_expert_gemm_fp4(
        torch.empty(0, K // 2, dtype=torch.uint8, device="cuda"), torch.empty(0, dtype=torch.uint8, device="cuda"),
        torch.empty(0, dtype=torch.float32, device="cuda"), to_dev(np.zeros(E + 1, np.int32)),
        torch.zeros(E, N, K // 2, dtype=torch.uint8, device="cuda"),
        torch.zeros(gpu.sf_swizzled_bytes(E * N, K // 16), dtype=torch.uint8, device="cuda"),
        torch.ones(E, dtype=torch.float32, device="cuda"), dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and out.shape[0] == 0


def test_gemm_all_experts_empty(gpu):
    """Capacity for 256 rows, but every expert received none: no tile is
    computed and the output buffer is left as it was."""
    E, N, K, M = 3, 256, 256, 256
    st = _status()
    out = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    gpu.grouped_expert_gemm_fp4(
        torch.zeros(M, K // 2, dtype=torch.uint8, device="cuda"),
        torch.zeros(gpu.sf_swizzled_bytes(M, K // 16), dtype=torch.uint8, device="cuda"),
        torch.ones(M, dtype=torch.float32, device="cuda"), to_dev(np.zeros(E + 1, np.int32)),
        torch.zeros(E, N, K // 2, dtype=torch.uint8, device="cuda"),
        torch.zeros(gpu.sf_swizzled_bytes(E * N, K // 16), dtype=torch.uint8, device="cuda"),
        torch.ones(E, dtype=torch.float32, device="cuda"), out=out, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert bool((out == 7.0).all())


def test_moe_no_tokens(gpu):
    E, H, I, k = 4, 256, 128, 2
    wgu = gpu.quantize_nvfp4_per_expert(torch.zeros(E, 2 * I, H, dtype=torch.bfloat16, device="cuda"))
    wd = gpu.quantize_nvfp4_per_expert(torch.zeros(E, H, I, dtype=torch.bfloat16, device="cuda"))
    st = _status()
    y = gpu.moe_expert_forward(torch.empty(0, H, dtype=torch.bfloat16, device="cuda"),
                               torch.empty(0, k, dtype=torch.int32, device="cuda"),
                               torch.empty(0, k, dtype=torch.float32, device="cuda"), wgu, wd, I, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and y.shape == (0, H)
