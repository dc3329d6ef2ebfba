"""Per-token NVFP4 of the 32-point random Hadamard transform against the
oracle, bit for bit: the in-register path (rows of up to 128 blocks) and the
two-pass path (longer rows), both scale-factor layouts, ragged row counts; and
the transform's effect on the outlier workload, reconstructed through the
inverse transform."""
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
@pytest.mark.parametrize("rows,K", [(300, 2048), (64, 96), (33, 4096), (16, 7168), (5, 32)])
def test_rht_matches_oracle(O, rows, K, swizzled):
    bsq = _bsq()
    x = synth.normal_with_outliers(rows, K, seed=rows + K)
    c, s, t = bsq.quantize_nvfp4_rht(to_dev(x), seed=7, swizzled=swizzled)
    rc, rs, rt = O.nvfp4_quantize_rht(x, seed=7)
    assert first_mismatch(to_np(t).view(np.uint32), rt.view(np.uint32)) is None
    assert first_mismatch(to_np(c), rc) is None, first_mismatch(to_np(c), rc)
    want_sf = O.sf_to_swizzled(rs) if swizzled else rs
    assert first_mismatch(to_np(s).reshape(want_sf.shape), want_sf) is None


def test_rht_zero_rows(O):
    bsq = _bsq()
    x = synth.normal_with_outliers(8, 256, seed=1)
    x[3] = 0
    c, s, t = bsq.quantize_nvfp4_rht(to_dev(x), seed=2)
    rc, rs, rt = O.nvfp4_quantize_rht(x, seed=2)
    assert to_np(t)[3] == 0.0 and not to_np(c)[3].any()
    assert first_mismatch(to_np(c), rc) is None


def test_rht_on_the_outlier_workload():
    # "End-to-End 4-Bit Training", "第三个决定": the transform spreads outliers
    # over their group.  Reconstruct x from the dequantized transform (s . H y
    # / 32) and compare with plain per-token NVFP4 of x on the requant
    # workload (1 % of the entries x20).
    bsq = _bsq()
    import scipy.linalg
    xh = synth.normal_with_outliers(16384, 2048, seed=7)
    x = to_dev(xh)
    xd = x.double()
    c, s, t = bsq.quantize_nvfp4_rht(x, seed=7)
    y = bsq.dequantize_nvfp4(c, s, t).double()
    import oracle
    signs = oracle.rht_signs(7)
    sg = torch.tensor(np.where((signs >> np.arange(32)) & 1, -1.0, 1.0), device="cuda", dtype=torch.float64)
    H = torch.tensor(scipy.linalg.hadamard(32), device="cuda", dtype=torch.float64)
    back = ((y.reshape(-1, 32) @ H.T) * sg / 32.0).reshape(xd.shape)
    c1, s1, t1 = bsq.quantize_nvfp4_per_token(x)
    plain = bsq.dequantize_nvfp4(c1, s1, t1).double()
    nz = xd != 0
    rel = {k: ((v - xd).norm() / xd.norm()).item() for k, v in (("rht", back), ("plain", plain))}
    flush = {k: ((v == 0) & nz).sum().item() / nz.sum().item() for k, v in (("rht", back), ("plain", plain))}
    for k in rel:
        print(f"{k:6s} relative RMS error {rel[k]:.4f}   nonzeros reconstructed as 0: {100 * flush[k]:.2f} %")
    # the transform is orthogonal up to 32: its quantization error maps back with the same norm scale
    assert rel["rht"] < 0.5 and rel["plain"] < 0.5
    assert flush["rht"] < flush["plain"]


def test_rht_boundary_rows(O):
    """Boundary rows (zeros, negative zeros, bf16 subnormals, E2M1 grid points
    and midpoints, one non-zero, a huge dynamic range; not the bf16 maximum,
    whose 32-term sums overflow), a constant row and a row of repeated pairs,
    whose butterfly sums cancel to exact zeros: the cross-lane stage's
    fma(+-1, v, o) keeps the sign of every zero the separate add and subtract
    give."""
    bsq = _bsq()
    sp = synth.special_rows(256)
    keep = [0, 1, 4, 5, 6, 7, 8]
    const = np.full((1, 256), synth.to_bf16_bits(np.array([1.5], np.float32))[0], np.uint16)
    pairs = np.repeat(synth.normal((1, 128), seed=5), 2, axis=1)
    x = np.concatenate([sp[keep], const, pairs]).astype(np.uint16)
    for swizzled in (False, True):
        c, s, t = bsq.quantize_nvfp4_rht(to_dev(x), seed=3, swizzled=swizzled)
        rc, rs, rt = O.nvfp4_quantize_rht(x, seed=3)
        assert first_mismatch(to_np(t).view(np.uint32), rt.view(np.uint32)) is None
        assert first_mismatch(to_np(c), rc) is None, first_mismatch(to_np(c), rc)
        want_sf = O.sf_to_swizzled(rs) if swizzled else rs
        assert first_mismatch(to_np(s).reshape(want_sf.shape), want_sf) is None
