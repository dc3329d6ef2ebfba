"""The Python binding without a GPU: every entry point rejects host (CPU)
tensors with BsqError before it reaches the library, so a product call can
never run on the host."""
import pytest
import torch

import block_scaled_precision_quantize_gb300 as bsq


def _u8(*shape):
    return torch.zeros(*shape, dtype=torch.uint8)


@pytest.mark.parametrize("call", [
    lambda: bsq.quantize_nvfp4_per_token(torch.zeros(4, 64, dtype=torch.bfloat16)),
    lambda: bsq.quantize_nvfp4_rht(torch.zeros(4, 64, dtype=torch.bfloat16)),
    lambda: bsq.quantize_nvfp4_2d(torch.zeros(16, 64, dtype=torch.bfloat16)),
    lambda: bsq.quantize_mxfp8_rowcol(torch.zeros(32, 64, dtype=torch.bfloat16)),
    lambda: bsq.dequantize_nvfp4(_u8(4, 32), _u8(4, 4), torch.ones(4)),
    lambda: bsq.grouped_expert_gemm_mxfp8(_u8(128, 128), _u8(128 * 4), torch.tensor([0, 128], dtype=torch.int32),
                                          _u8(1, 128, 128), _u8(128 * 4)),
    lambda: bsq.grouped_expert_gemm_fp4(_u8(128, 64), _u8(128 * 8), torch.ones(128),
                                        torch.tensor([0, 128], dtype=torch.int32), _u8(1, 128, 64), _u8(128 * 8),
                                        torch.ones(1)),
])
def test_host_tensors_are_rejected(call):
    with pytest.raises(bsq.BsqError, match="CUDA tensor"):
        call()
