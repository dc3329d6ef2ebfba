"""GPU: the quantizer kernels against the oracle, bit-exact (codes, scale
bytes and FP32 scales), on random, outlier, boundary, all-zero and
maximum-value tensors, ragged shapes, both SF layouts, and the full-size
workloads."""
import numpy as np
import pytest
import torch

from block_scaled_precision_quantize_gb300 import synth
from conftest import bits_equal, first_mismatch, to_dev, to_np

pytestmark = pytest.mark.gpu


def _check(got, ref, what):
    assert bits_equal(got, ref), f"{what}: {first_mismatch(got, ref)}"


def _nvfp4_case(gpu, O, x, four_six, swz):
    codes, sf, t = gpu.quantize_nvfp4_per_token(to_dev(x), four_six=four_six, swizzled=swz)
    oc, osf, ot = O.nvfp4_quantize_rows(x, four_six=four_six)
    _check(to_np(codes), oc, "codes")
    _check(to_np(t), ot, "row scale")
    _check(to_np(sf), O.sf_to_swizzled(osf) if swz else osf, "sf")


@pytest.mark.parametrize("rows,K", [(64, 256), (300, 2048), (37, 7168), (5, 16), (129, 12288), (64, 1040),
                                    (1, 8192), (200, 768)])
@pytest.mark.parametrize("four_six", [False, True])
@pytest.mark.parametrize("swz", [False, True])
def test_nvfp4_per_token(gpu, O, rows, K, four_six, swz):
    x = synth.normal_with_outliers(rows, K, seed=rows * 7 + K)
    _nvfp4_case(gpu, O, x, four_six, swz)


@pytest.mark.parametrize("swz", [False, True])
def test_nvfp4_four_six_tie(gpu, O, swz):
    """Rows holding the block whose two 4/6 candidates tie in binary32 (the
    oracle pin of the same name): the kernel keeps the 6-candidate too."""
    from test_oracle_quant import four_six_tie_row
    tie = four_six_tie_row()
    x = synth.normal_with_outliers(96, 256, seed=5)
    x[::3, :32] = tie
    x[1::3, 224:] = tie
    _nvfp4_case(gpu, O, x, True, swz)


@pytest.mark.parametrize("four_six", [False, True])
def test_nvfp4_boundary_rows(gpu, O, four_six):
    x = synth.special_rows(512)
    wide = synth.rows_log_uniform_std(64, 512, seed=3, lo_exp=-30, hi_exp=30)
    _nvfp4_case(gpu, O, np.concatenate([x, wide]), four_six, True)


def test_nvfp4_all_zero_and_max(gpu, O):
    x = np.zeros((32, 256), np.uint16)
    x[16:] = 0x7F7F
    x[20:, ::3] = 0xFF7F
    _nvfp4_case(gpu, O, x, True, False)


def test_nvfp4_empty(gpu):
    x = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    codes, sf, t = gpu.quantize_nvfp4_per_token(x)
    assert codes.numel() == 0 and t.numel() == 0


def test_nvfp4_batch_invariance_on_gpu(gpu):
    x = synth.normal_with_outliers(96, 2048, seed=31)
    c0, s0, t0 = gpu.quantize_nvfp4_per_token(to_dev(x))
    c1, s1, t1 = gpu.quantize_nvfp4_per_token(to_dev(x[40:41]))
    assert torch.equal(c0[40:41], c1) and torch.equal(s0[40:41], s1) and torch.equal(t0[40:41], t1)


@pytest.mark.parametrize("E,rows,K", [(3, 256, 128), (2, 128, 2048), (4, 130, 64)])
@pytest.mark.parametrize("swz", [False, True])
def test_nvfp4_per_expert(gpu, O, E, rows, K, swz):
    if swz and rows % 128:
        pytest.skip("swizzled weights need rows % 128 == 0")
    w = synth.normal((E, rows, K), seed=E + rows, std=0.02)
    codes, sf, t = gpu.quantize_nvfp4_per_expert(to_dev(w), swizzled=swz)
    oc, osf, ot = O.nvfp4_quantize_group(w)
    _check(to_np(codes), oc, "codes")
    _check(to_np(t), ot, "expert scale")
    ref_sf = O.sf_to_swizzled(osf.reshape(E * rows, K // 16)) if swz else osf
    _check(to_np(sf), ref_sf, "sf")


@pytest.mark.parametrize("rows,K", [(64, 256), (96, 160), (256, 2048), (32, 32), (160, 4096)])
@pytest.mark.parametrize("swz", [False, True])
def test_mxfp8_rowcol(gpu, O, rows, K, swz):
    x = synth.rows_log_uniform_std(rows, K, seed=rows + K)
    rc, rs, cc, cs = gpu.quantize_mxfp8_rowcol(to_dev(x), swizzled=swz)
    orc, ors, occ, ocs = O.mxfp8_quantize_rowcol(x)
    _check(to_np(rc), orc, "row codes")
    _check(to_np(cc), occ, "col codes")
    _check(to_np(rs), O.sf_to_swizzled(ors) if swz else ors, "row sf")
    _check(to_np(cs), O.sf_to_swizzled(ocs) if swz else ocs, "col sf")


def test_mxfp8_one_copy_only(gpu, O):
    x = synth.normal_with_outliers(64, 128, seed=5)
    rc, rs, cc, cs = gpu.quantize_mxfp8_rowcol(to_dev(x), col=False)
    assert cc is None
    orc, ors, occ, ocs = O.mxfp8_quantize_rowcol(x)
    _check(to_np(rc), orc, "row codes")
    rc, rs, cc, cs = gpu.quantize_mxfp8_rowcol(to_dev(x), row=False)
    _check(to_np(cc), occ, "col codes")
    _check(to_np(cs), ocs, "col sf")


def test_mxfp8_boundary(gpu, O):
    x = np.concatenate([synth.special_rows(256), np.zeros((23, 256), np.uint16)])
    rc, rs, cc, cs = gpu.quantize_mxfp8_rowcol(to_dev(x))
    orc, ors, occ, ocs = O.mxfp8_quantize_rowcol(x)
    for g, r, n in ((rc, orc, "rc"), (rs, ors, "rs"), (cc, occ, "cc"), (cs, ocs, "cs")):
        _check(to_np(g), r, n)


def _requant_inputs(O, rows, K, seed):
    x = synth.normal_with_outliers(rows, K, seed=seed)
    return O.nvfp4_quantize_rows(x)


@pytest.mark.parametrize("rows,K", [(64, 96), (160, 2048), (1024, 768), (32, 16), (64, 48), (96, 80), (288, 176)])
@pytest.mark.parametrize("sr", [False, True])
@pytest.mark.parametrize("swz", [False, True])
def test_requant_transpose(gpu, O, rows, K, sr, swz):
    codes, sf, t = _requant_inputs(O, rows, K, seed=rows + K)
    sf_in = O.sf_to_swizzled(sf) if swz else sf
    out = gpu.requant_transpose_sr(to_dev(codes), to_dev(sf_in), to_dev(t), stochastic=sr, seed=7, swizzled=swz)
    nc, ns, nt, mc, ms = O.requant_transpose(codes, sf, t, sr=sr, seed=7)
    _check(to_np(out["nv_codes"]), nc, "nvfp4 codes")
    _check(to_np(out["nv_scale"]), nt, "nvfp4 scale")
    _check(to_np(out["nv_sf"]), O.sf_to_swizzled(ns) if swz else ns, "nvfp4 sf")
    _check(to_np(out["mx_codes"]), mc, "mxfp8 codes")
    _check(to_np(out["mx_sf"]), O.sf_to_swizzled(ms) if swz else ms, "mxfp8 sf")


def test_requant_single_targets(gpu, O):
    codes, sf, t = _requant_inputs(O, 96, 256, seed=3)
    nc, ns, nt, mc, ms = O.requant_transpose(codes, sf, t, sr=True, seed=11)
    o1 = gpu.requant_transpose_sr(to_dev(codes), to_dev(sf), to_dev(t), mxfp8=False, seed=11)
    assert o1["mx_codes"] is None
    _check(to_np(o1["nv_codes"]), nc, "nv only")
    o2 = gpu.requant_transpose_sr(to_dev(codes), to_dev(sf), to_dev(t), nvfp4=False, seed=11)
    assert o2["nv_codes"] is None
    _check(to_np(o2["mx_codes"]), mc, "mx only")


def test_requant_page_example_on_gpu(gpu, O):
    """The page's 4.5 -> (scale 2) -> 2.25 -> SR {2: 3/4, 3: 1/4} example
    through the CUDA requant, over 10^6 draws, bit-exact with the oracle."""
    M = 1066688
    codes = np.zeros((M, 8), np.uint8)
    sf = np.full((M, 1), 0x51, np.uint8)
    codes[:, 0] = 0x1
    codes[::16, 0] = 0x7
    sf[::16, 0] = 0x40
    t = np.ones(M, np.float32)
    out = gpu.requant_transpose_sr(to_dev(codes), to_dev(sf), to_dev(t), mxfp8=False, stochastic=True, seed=7)
    nc, ns, nt, _, _ = O.requant_transpose(codes, sf, t, sr=True, seed=7, mxfp8=False)
    _check(to_np(out["nv_codes"]), nc, "codes")
    row = to_np(out["nv_codes"])[0]
    lo = row & 0xF
    hi = row >> 4
    nib = np.stack([lo, hi], axis=1).ravel()
    sel = np.ones(M, bool)
    sel[::16] = False
    p3 = np.mean(nib[sel] == 0x5)
    assert abs(p3 - 0.25) < 0.005 and set(np.unique(nib[sel])) == {0x4, 0x5}


def _requant_scale_edge_inputs():
    """An NVFP4 input whose transposed rows exercise the block-scale quotient
    amax / rn(6 t) at its edges.  Columns 0..15: row 0 sets every column
    maximum to 2688 (E2M1 6 x E4M3 448 x t 1), so t = 1 and rn(6 t) = 6; in
    the second, third and fourth 16-row blocks one row each holds E2M1 codes
    c times scale s = 6.375, 6.375 (1 + 2^-22), 6.375 (1 - 2^-22): the
    quotient is c * 1.0625 (exactly an E4M3 rounding midpoint for c = 0.5, 1,
    2, 4: ties to even) or within 2^-20 of it.  Columns 16..31: one row with
    t = 1e-38, so the column maximum is 6e-38 and 1 / rn(6 t) overflows."""
    rows, K = 64, 32
    codes = np.zeros((rows, K // 2), np.uint8)
    sf = np.zeros((rows, K // 16), np.uint8)
    t = np.zeros(rows, np.float32)

    def put(r, k, code):
        b = int(codes[r, k // 2])
        codes[r, k // 2] = (b & 0xF0) | code if k % 2 == 0 else (b & 0x0F) | (code << 4)

    t[0], sf[0, 0] = 1.0, 0x7E
    for k in range(16):
        put(0, k, 0x7)
    mags = [1, 2, 4, 6, 3, 5, 7, 0x9, 0xA, 0xC, 0xE]  # 0.5, 1, 2, 4 (ties), 1.5, 3, 6, negatives
    for r, s in ((16, 6.375), (32, 6.375 * (1 + 2.0 ** -22)), (48, 6.375 * (1 - 2.0 ** -22))):
        t[r], sf[r, 0] = np.float32(s), 0x38
        for k in range(16):
            put(r, k, mags[(k + r) % len(mags)])
    t[1], sf[1, 1] = np.float32(1e-38), 0x38
    for k in range(16, 32):
        put(1, k, mags[k % len(mags)])
    return codes, sf, t


@pytest.mark.parametrize("sr", [False, True])
@pytest.mark.parametrize("swz", [False, True])
def test_requant_block_scale_quotient_edges(gpu, O, sr, swz):
    codes, sf, t = _requant_scale_edge_inputs()
    sf_in = O.sf_to_swizzled(sf) if swz else sf
    out = gpu.requant_transpose_sr(to_dev(codes), to_dev(sf_in), to_dev(t), stochastic=sr, seed=5, swizzled=swz)
    nc, ns, nt, mc, ms = O.requant_transpose(codes, sf, t, sr=sr, seed=5)
    _check(to_np(out["nv_scale"]), nt, "nvfp4 scale")
    _check(to_np(out["nv_sf"]), O.sf_to_swizzled(ns) if swz else ns, "nvfp4 sf")
    _check(to_np(out["nv_codes"]), nc, "nvfp4 codes")
    _check(to_np(out["mx_codes"]), mc, "mxfp8 codes")
    _check(to_np(out["mx_sf"]), O.sf_to_swizzled(ms) if swz else ms, "mxfp8 sf")


@pytest.mark.parametrize("shape", [(16384, 2048), (16384, 768)])
def test_requant_full_size(gpu, O, shape):
    """The backward-requant workload at full size, SR seed 7, bit-exact."""
    rows, K = shape
    x = synth.normal_with_outliers(rows, K, seed=7)
    codes, sf, t = O.nvfp4_quantize_rows(x)
    out = gpu.requant_transpose_sr(to_dev(codes), to_dev(O.sf_to_swizzled(sf)), to_dev(t), stochastic=True,
                                   seed=7, swizzled=True)
    nc, ns, nt, mc, ms = O.requant_transpose(codes, sf, t, sr=True, seed=7)
    _check(to_np(out["nv_codes"]), nc, "nvfp4 codes")
    _check(to_np(out["nv_sf"]), O.sf_to_swizzled(ns), "nvfp4 sf")
    _check(to_np(out["nv_scale"]), nt, "nvfp4 scale")
    _check(to_np(out["mx_codes"]), mc, "mxfp8 codes")
    _check(to_np(out["mx_sf"]), O.sf_to_swizzled(ms), "mxfp8 sf")


def test_mxfp8_full_size(gpu, O):
    """The MXFP8 row+column workload (16384 x 2048, row std 10^U(-3,2))."""
    x = synth.rows_log_uniform_std(16384, 2048, seed=2)
    rc, rs, cc, cs = gpu.quantize_mxfp8_rowcol(to_dev(x))
    orc, ors, occ, ocs = O.mxfp8_quantize_rowcol(x)
    for g, r, n in ((rc, orc, "rc"), (rs, ors, "rs"), (cc, occ, "cc"), (cs, ocs, "cs")):
        _check(to_np(g), r, n)


def test_nvfp4_full_size_activations(gpu, O):
    x = synth.normal(( 16384, 2048), seed=3)
    _nvfp4_case(gpu, O, x, False, True)
