"""Parity of the BF16 dequantization (the operands of the dequantized
backward mode) with the oracle, bit for bit: per-token and per-expert
scales, linear and swizzled block scales, ragged shapes (K not a multiple of
64 takes the one-block-per-thread path), output rows with a pitch, zero
scales and empty inputs, and the full 16384 x 2048 launch on sampled rows."""
import numpy as np
import pytest
import torch

from block_scaled_precision_quantize_gb300 import synth
from conftest import first_mismatch, to_dev, to_np

pytestmark = pytest.mark.gpu


def _bsq():
    import block_scaled_precision_quantize_gb300 as bsq
    bsq.build()
    return bsq


@pytest.mark.parametrize("swizzled", [False, True])
@pytest.mark.parametrize("rows,K", [(300, 2048), (129, 80), (1, 16), (256, 768)])
def test_dequant_per_token(O, rows, K, swizzled):
    bsq = _bsq()
    codes, sf, t = synth.random_nvfp4(rows, K, seed=rows + K)
    sf_in = O.sf_to_swizzled(sf) if swizzled else sf
    y = bsq.dequantize_nvfp4(to_dev(codes), to_dev(sf_in), to_dev(t), swizzled=swizzled)
    got, ref = to_np(y), O.nvfp4_dequantize_bf16(codes, sf, t)
    assert first_mismatch(got, ref) is None, first_mismatch(got, ref)


@pytest.mark.parametrize("swizzled", [False, True])
def test_dequant_per_expert(O, swizzled):
    bsq = _bsq()
    E, N, K = 3, 256, 512
    codes, sf, t = synth.random_nvfp4(E * N, K, seed=5, groups=E)
    sf_in = O.sf_to_swizzled(sf) if swizzled else sf
    y = bsq.dequantize_nvfp4(to_dev(codes.reshape(E, N, K // 2)), to_dev(sf_in), to_dev(t), swizzled=swizzled)
    assert tuple(y.shape) == (E, N, K)
    got, ref = to_np(y).reshape(E * N, K), O.nvfp4_dequantize_bf16(codes, sf, np.repeat(t, N))
    assert first_mismatch(got, ref) is None, first_mismatch(got, ref)


@pytest.mark.parametrize("pad", [64, 8])  # row pitch a multiple of 16 elements (256-bit stores) or only of 8
def test_dequant_into_pitched_rows(O, pad):
    bsq = _bsq()
    rows, K = 200, 1024
    codes, sf, t = synth.random_nvfp4(rows, K, seed=8)
    buf = torch.full((rows, K + pad), -1.0, dtype=torch.bfloat16, device="cuda")
    bsq.dequantize_nvfp4(to_dev(codes), to_dev(sf), to_dev(t), y=buf[:, :K])
    got, ref = to_np(buf[:, :K]), O.nvfp4_dequantize_bf16(codes, sf, t)
    assert first_mismatch(got, ref) is None, first_mismatch(got, ref)
    assert bool((buf[:, K:] == -1.0).all())


def test_dequant_zero_scales_and_empty(O):
    bsq = _bsq()
    codes, sf, t = synth.random_nvfp4(64, 256, seed=9)
    t[::2] = 0.0
    y = bsq.dequantize_nvfp4(to_dev(codes), to_dev(sf), to_dev(t))
    got, ref = to_np(y), O.nvfp4_dequantize_bf16(codes, sf, t)
    assert first_mismatch(got, ref) is None, first_mismatch(got, ref)
    assert not (got[::2] & 0x7FFF).any()  # zero rows: +-0 only
    e = bsq.dequantize_nvfp4(torch.empty(0, 128, dtype=torch.uint8, device="cuda"),
                             torch.empty(0, 16, dtype=torch.uint8, device="cuda"),
                             torch.empty(0, dtype=torch.float32, device="cuda"))
    assert tuple(e.shape) == (0, 256)


def test_dequant_full_size_sampled(O):
    # the bench's launch: 16384 x 2048, swizzled block scales
    bsq = _bsq()
    rows, K = 16384, 2048
    codes, sf, t = synth.random_nvfp4(rows, K, seed=12)
    y = bsq.dequantize_nvfp4(to_dev(codes), to_dev(O.sf_to_swizzled(sf)), to_dev(t), swizzled=True)
    pick = np.concatenate([[0, 127, 128, rows - 1], np.random.default_rng(0).choice(rows, 60, replace=False)])
    got, ref = to_np(y)[pick], O.nvfp4_dequantize_bf16(codes[pick], sf[pick], t[pick])
    assert first_mismatch(got, ref) is None, first_mismatch(got, ref)
