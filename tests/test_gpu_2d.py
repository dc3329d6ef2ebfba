"""2-D NVFP4 (16 x 16 block scales, one FP32 scale per tensor) against the
oracle, bit for bit, for both the row-major and the transposed operand, on
ragged shapes and the full 16384 x 2048 backward workload; and the page's
comparison of square block scales with the requantize route on that
workload."""
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


def _check_against_oracle(O, x, got):
    c, s, ct, st, t = got
    rc, rs, rt = O.nvfp4_quantize_2d(x)
    rcT, rsT, rtT = O.nvfp4_quantize_2d(np.ascontiguousarray(x.T))
    assert np.float32(rt) == np.float32(rtT)
    assert to_np(t).view(np.uint32)[0] == np.array([rt], np.float32).view(np.uint32)[0]
    for name, a, b in (("codes", to_np(c), rc), ("sf", to_np(s), rs)):
        assert first_mismatch(a, b) is None, (name, first_mismatch(a, b))
    if ct is not None:
        for name, a, b in (("codes_t", to_np(ct), rcT), ("sf_t", to_np(st), rsT)):
            assert first_mismatch(a, b) is None, (name, first_mismatch(a, b))


@pytest.mark.parametrize("rows,K", [(256, 2048), (48, 80), (16, 16), (64, 272)])
def test_2d_matches_oracle(O, rows, K):
    bsq = _bsq()
    x = synth.normal_with_outliers(rows, K, seed=rows + K)
    _check_against_oracle(O, x, bsq.quantize_nvfp4_2d(to_dev(x)))


def test_2d_row_operand_only_and_zero_tensor(O):
    bsq = _bsq()
    x = synth.normal_with_outliers(64, 512, seed=3)
    got = bsq.quantize_nvfp4_2d(to_dev(x), transposed=False)
    assert got[2] is None and got[3] is None
    _check_against_oracle(O, x, got)
    z = np.zeros((32, 64), np.uint16)
    c, s, ct, st, t = bsq.quantize_nvfp4_2d(to_dev(z))
    assert float(t.item()) == 0.0
    assert not to_np(c).any() and not to_np(s).any() and not to_np(ct).any() and not to_np(st).any()


def test_2d_full_size(O):
    # the backward workload: 16384 x 2048 bf16 ~N(0,1) with 1% of entries x20
    bsq = _bsq()
    x = synth.normal_with_outliers(16384, 2048, seed=7)
    _check_against_oracle(O, x, bsq.quantize_nvfp4_2d(to_dev(x)))


def _dequant_t(bsq, codes_t, sf_rows, scale_rows):
    return bsq.dequantize_nvfp4(codes_t, sf_rows.contiguous(), scale_rows.contiguous()).double()


def test_2d_against_requantize_on_the_backward_workload():
    # "End-to-End 4-Bit Training", "第二个决定": square 16 x 16 scales keep the
    # transposed operand free of requantization, but one outlier among 256
    # values flushes the others; the requantize route (1 x 16 forward,
    # dequantize, transpose, requantize with stochastic rounding) keeps far
    # more of the small values.  Both transposed operands are compared with
    # x^T, next to quantizing x^T directly (not available in the backward pass).
    bsq = _bsq()
    x = to_dev(synth.normal_with_outliers(16384, 2048, seed=7))
    xt = x.t().contiguous().double()
    K, rows = xt.shape
    res = {}
    _, _, ct, st, t = bsq.quantize_nvfp4_2d(x)
    res["2-D 16x16"] = _dequant_t(bsq, ct, st.repeat_interleave(16, dim=0), t.expand(K))
    c1, s1, t1 = bsq.quantize_nvfp4_per_token(x)
    for sr in (True, False):
        r = bsq.requant_transpose_sr(c1, s1, t1, nvfp4=True, mxfp8=False, stochastic=sr, seed=7)
        res["requant " + ("SR" if sr else "RNE")] = _dequant_t(bsq, r["nv_codes"], r["nv_sf"], r["nv_scale"])
    cd, sd, td = bsq.quantize_nvfp4_per_token(x.t().contiguous())
    res["1x16 of x^T"] = _dequant_t(bsq, cd, sd, td)
    nz = xt != 0
    stats = {}
    for k, y in res.items():
        flush = ((y == 0) & nz).sum().item() / nz.sum().item()
        rel = ((y - xt).norm() / xt.norm()).item()
        stats[k] = (flush, rel)
        print(f"{k:14s} nonzeros flushed to 0: {100 * flush:6.2f} %   relative RMS error: {rel:.4f}")
    assert stats["2-D 16x16"][0] > 2 * stats["requant SR"][0]
    assert stats["2-D 16x16"][1] > stats["requant SR"][1]
    assert stats["1x16 of x^T"][1] <= stats["requant SR"][1]


def test_2d_boundary_rows(O):
    """Boundary rows (zeros, negative zeros, the bf16 maximum with both signs,
    subnormals, E2M1 grid points, one non-zero, a huge dynamic range) in
    16-row tiles: the tile maximum is taken on packed bf16 magnitudes."""
    bsq = _bsq()
    sp = synth.special_rows(96)
    x = np.concatenate([np.repeat(sp, 2, axis=0), sp[::-1]]).astype(np.uint16)[:16 * (27 // 16 + 1)]
    x = np.concatenate([x, np.zeros((32 - x.shape[0] % 32 if x.shape[0] % 32 else 0, 96), np.uint16)])
    _check_against_oracle(O, x, bsq.quantize_nvfp4_2d(to_dev(x)))
    # the tiles without the bf16 maximum (its tensor scale would flush them)
    y = np.concatenate([sp[[0, 1, 4, 5, 6, 7, 8]]] * 3)[:16]
    _check_against_oracle(O, y, bsq.quantize_nvfp4_2d(to_dev(y)))
