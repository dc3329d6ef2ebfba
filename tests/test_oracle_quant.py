"""Oracle pins for the NVFP4 / MXFP8 quantizers and the backward requant:
page examples, invariants, closed forms and library cross-checks (CPU)."""
import math

import numpy as np
import pytest
import torch

from conftest import golden
from block_scaled_precision_quantize_gb300 import synth

PAGE = golden("page_examples.json")
E2M1 = np.array(PAGE["nvfp4_value_set"]["magnitudes"] + [-m for m in PAGE["nvfp4_value_set"]["magnitudes"]])


def e2m1_val(codes):
    c = np.asarray(codes, np.int64)
    return E2M1[(c & 7) + 8 * ((c >> 3) & 1)]


def unpack(codes):
    c = np.asarray(codes, np.uint8)
    out = np.empty(c.shape[:-1] + (c.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = c & 0xF
    out[..., 1::2] = c >> 4
    return out


def e4m3_val(b):
    return torch.from_numpy(np.asarray(b, np.uint8).copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_neg54_is_minus6_times_9(O):
    ex = PAGE["neg54_block_scale"]
    x = np.zeros((1, 16), np.float32)
    x[0, 3] = ex["value"]
    x[0, 7] = 1.0
    codes, sf = O.nvfp4_quantize_rows_given_t(x, np.array([1.0], np.float32))
    assert O.e4m3_decode(sf[0, 0]) == ex["block_scale"]
    assert O.e2m1_decode(unpack(codes)[0, 3]) == ex["element"]
    assert unpack(codes)[0, 3] == 0xF


def test_forward_5p4_becomes_4p5_under_scale_9(O):
    ex = PAGE["requant_example"]
    x = np.zeros((1, 16), np.float32)
    x[0, 0] = 54.0                 # block amax 54 -> scale 9
    x[0, 5] = ex["forward_value"]
    codes, sf = O.nvfp4_quantize_rows_given_t(x, np.array([1.0], np.float32))
    assert O.e4m3_decode(sf[0, 0]) == ex["forward_scale"]
    deq = O.nvfp4_dequantize(codes, sf, np.array([1.0], np.float32))
    assert deq[0, 5] == ex["forward_dequant"]


def test_requant_4p5_under_scale_2_rne(O):
    ex = PAGE["requant_example"]
    x = np.zeros((1, 16), np.float32)
    x[0, 0] = 12.0                 # block amax 12 -> scale 2
    x[0, 9] = ex["forward_dequant"]
    codes, sf = O.nvfp4_quantize_rows_given_t(x, np.array([1.0], np.float32))
    assert O.e4m3_decode(sf[0, 0]) == ex["new_scale"]
    assert O.e2m1_decode(unpack(codes)[0, 9]) == ex["rne_element"]
    deq = O.nvfp4_dequantize(codes, sf, np.array([1.0], np.float32))
    assert deq[0, 9] == ex["rne_dequant"]


def _requant_example_input(M):
    """NVFP4 [M, 16] tensor whose column 0 dequantizes to 4.5 (= 0.5 x scale
    9, the page's forward result) except every 16th row, which holds 12
    (= 6 x scale 2) so that each 16-block of the transposed row has amax 12."""
    codes = np.zeros((M, 8), np.uint8)
    sf = np.full((M, 1), 0x51, np.uint8)          # E4M3 9.0
    codes[:, 0] = 0x1                              # 0.5
    codes[::16, 0] = 0x7                           # 6
    sf[::16, 0] = 0x40                             # E4M3 2.0
    t = np.ones(M, np.float32)
    return codes, sf, t


def test_requant_sr_example_over_a_million_draws(O):
    ex = PAGE["requant_example"]
    M = 1066688                                     # 15/16 of it >= 10^6 draws of 4.5
    codes, sf, t = _requant_example_input(M)
    deq_in = O.nvfp4_dequantize(codes[:32], sf[:32], t[:32])
    assert deq_in[1, 0] == 4.5 and deq_in[0, 0] == 12.0
    for sr in (False, True):
        nc, ns, nt, _, _ = O.requant_transpose(codes, sf, t, sr=sr, seed=ex["seed"], mxfp8=False)
        row = unpack(nc[0:1])[0]                    # transposed column 0
        d = e4m3_val(ns[0]).repeat(16) * np.float64(nt[0])
        vals = e2m1_val(row) * d
        sel = np.ones(M, bool)
        sel[::16] = False
        assert sel.sum() >= ex["draws"]
        # the block scale came out as the page's 2 (up to the FP32 scale's rounding)
        assert abs(d[1] - ex["new_scale"]) < 1e-6
        el = e2m1_val(row[sel])
        if not sr:
            assert np.all(el == ex["rne_element"])
        else:
            assert set(np.unique(el)) == {ex["sr_low"], ex["sr_high"]}
            p_hi = np.mean(el == ex["sr_high"])
            assert abs(p_hi - ex["p_high"]) < 0.005
            mean = vals[sel].mean()
            assert abs(mean - ex["expected_dequant"]) / ex["expected_dequant"] < ex["rel_tol"]


def test_bits_per_value(O):
    bpv = PAGE["bits_per_value"]
    x = synth.normal((64, 256), seed=1)
    codes, sf, t = O.nvfp4_quantize_rows(x)
    assert (codes.nbytes + sf.nbytes) * 8 / x.size == bpv["nvfp4"]
    rc, rs, cc, cs = O.mxfp8_quantize_rowcol(x)
    assert (rc.nbytes + rs.nbytes) * 8 / x.size == bpv["mxfp8"]
    assert (cc.nbytes + cs.nbytes) * 8 / x.size == bpv["mxfp8"]
    assert x.dtype.itemsize * 8 == bpv["bf16"]
    assert sf.shape[1] * PAGE["block_sizes"]["nvfp4_block"] == x.shape[1]
    assert rs.shape[1] * PAGE["block_sizes"]["mxfp8_block"] == x.shape[1]


def test_nvfp4_scale_and_codes_closed_form(O):
    # per-token scale t = amax / 2688; largest block scale lands at 448
    x = synth.normal_with_outliers(32, 512, seed=5)
    codes, sf, t = O.nvfp4_quantize_rows(x)
    xf = synth.bf16_bits_to_f32(x)
    amax = np.abs(xf).max(axis=1)
    assert np.array_equal(t, (amax / np.float32(2688)).astype(np.float32))
    assert np.all(sf.max(axis=1) == 0x7E)
    # dequantized values stay within half a grid step of the input
    deq = O.nvfp4_dequantize(codes, sf, t).astype(np.float64)
    d = (e4m3_val(sf) * t[:, None].astype(np.float64)).repeat(16, axis=1)
    assert np.all(np.abs(deq - xf) <= d * 1.0 + 1e-30)   # <= half of the widest step (2 x d / 2)


def test_zero_and_degenerate_rows(O):
    x = synth.special_rows(256)
    codes, sf, t = O.nvfp4_quantize_rows(x)
    assert t[0] == 0 and not codes[0].any() and not sf[0].any()
    assert t[1] == 0 and not codes[1].any() and not sf[1].any()          # all -0.0
    assert np.isfinite(t).all()
    # the bf16 maximum row: every element is +-6 with scale 448
    assert np.all(sf[2] == 0x7E) and np.all(unpack(codes[2:3]) == 0x7)
    assert np.all(unpack(codes[3:4])[0, 1::2] == 0xF)


def test_per_token_batch_invariance(O):
    x = synth.normal_with_outliers(48, 384, seed=9)
    codes, sf, t = O.nvfp4_quantize_rows(x)
    perm = np.random.default_rng(0).permutation(48)
    pc, ps, pt = O.nvfp4_quantize_rows(x[perm])
    assert np.array_equal(pc, codes[perm]) and np.array_equal(ps, sf[perm]) and np.array_equal(pt, t[perm])
    other = synth.normal(( 16, 384), seed=99, std=1000.0)
    mix = np.concatenate([x[:5], other])
    mc, ms, mt = O.nvfp4_quantize_rows(mix)
    assert np.array_equal(mc[:5], codes[:5]) and np.array_equal(ms[:5], sf[:5]) and np.array_equal(mt[:5], t[:5])
    for i in (0, 17, 47):
        c1, s1, t1 = O.nvfp4_quantize_rows(x[i:i + 1])
        assert np.array_equal(c1[0], codes[i]) and np.array_equal(s1[0], sf[i]) and t1[0] == t[i]


@pytest.mark.parametrize("k", [-20, -3, 1, 7, 30])
def test_power_of_two_scale_invariance(O, k):
    x = synth.normal_with_outliers(32, 256, seed=4)
    xf = synth.bf16_bits_to_f32(x)
    xs = synth.to_bf16_bits(xf * np.float32(2.0 ** k))
    assert np.array_equal(synth.bf16_bits_to_f32(xs), xf * np.float32(2.0 ** k))   # exact
    c0, s0, t0 = O.nvfp4_quantize_rows(x)
    c1, s1, t1 = O.nvfp4_quantize_rows(xs)
    assert np.array_equal(c0, c1) and np.array_equal(s0, s1)
    assert np.array_equal(t1, t0 * np.float32(2.0 ** k))
    r0 = O.mxfp8_quantize_rowcol(x)
    r1 = O.mxfp8_quantize_rowcol(xs)
    assert np.array_equal(r0[0], r1[0]) and np.array_equal(r0[2], r1[2])
    nz = r0[1] != 0
    assert np.array_equal(r1[1][nz].astype(int), r0[1][nz].astype(int) + k)


def test_group_scale_is_one_per_expert(O):
    w = synth.normal((3, 256, 128), seed=6, std=0.02)
    codes, sf, t = O.nvfp4_quantize_group(w)
    wf = synth.bf16_bits_to_f32(w)
    for g in range(3):
        assert t[g] == np.float32(np.abs(wf[g]).max()) / np.float32(2688)
        c2, s2 = O.nvfp4_quantize_rows_given_t(wf[g], np.full(256, t[g], np.float32))
        assert np.array_equal(c2, codes[g]) and np.array_equal(s2, sf[g])


def test_four_six_brute_force(O):
    """4/6 picks, per block, the candidate with the smaller error; checked in
    fp64 against both candidates, and never worse than the 6-only recipe."""
    x = synth.normal_with_outliers(64, 256, seed=21)
    xf = synth.bf16_bits_to_f32(x).astype(np.float32)
    c6, s6, t = O.nvfp4_quantize_rows(x, four_six=False)
    c46, s46, t46 = O.nvfp4_quantize_rows(x, four_six=True)
    assert np.array_equal(t, t46)
    n_four = 0
    for r in range(64):
        for b in range(16):
            blk = xf[r, 16 * b:16 * b + 16]
            cand = {}
            for m in (6.0, 4.0):
                cc, ss, sse32 = O.nvfp4_block_candidate(blk, t[r], m)
                d = np.float64(np.float32(e4m3_val([ss])[0] * np.float64(t[r])))
                rec = e2m1_val(cc) * d
                cand[m] = (cc, ss, float(np.sum((blk.astype(np.float64) - rec) ** 2)), sse32)
            chosen = unpack(c46[r:r + 1, 8 * b:8 * b + 8])[0]
            pick = 4.0 if (np.array_equal(chosen, cand[4.0][0]) and s46[r, b] == cand[4.0][1]
                           and not (np.array_equal(chosen, cand[6.0][0]) and s46[r, b] == cand[6.0][1])) else 6.0
            n_four += pick == 4.0
            e6, e4 = cand[6.0][2], cand[4.0][2]
            margin = 1e-5 * max(e6, e4) + 1e-30
            if e4 < e6 - margin:
                assert pick == 4.0
            elif e6 < e4 - margin:
                assert pick == 6.0
            assert cand[pick][2] <= min(e6, e4) + margin
            if pick == 6.0:
                assert np.array_equal(chosen, unpack(c6[r:r + 1, 8 * b:8 * b + 8])[0]) and s6[r, b] == s46[r, b]
    assert n_four > 50   # the second candidate does get used on N(0,1) data


# A block with one outlier (28.5) among small values, in a row whose maximum
# (50.75, in the first block) sets t = rn(50.75 / 2688).  The candidates' block
# scales are 256 (the 6-candidate) and 384 (the 4-candidate).  Both encode
# 28.5 as 6 x 4.8333335 = 29 and 4 x 7.25 = 29 in binary32, and every other
# element as 0, so the binary32 error sums tie and the strict rule keeps the
# 6-candidate.  In exact arithmetic, or with the multiply and the subtract
# fused, 6 x 4.8333335 is 29.000001 and the 4-candidate would look better: the
# case pins the per-operation rounding of the error sum.
FOUR_SIX_TIE_BLOCK = [-0.6484375, -0.8046875, -1.078125, -0.6484375, -0.7578125, -0.91796875, -0.1845703125,
                      -1.140625, 0.052978515625, 0.31640625, -0.498046875, -0.97265625, 28.5, 0.85546875,
                      -0.052734375, 0.1572265625]


def four_six_tie_row():
    row = np.zeros(32, np.float32)
    row[0] = 50.75
    row[16:] = FOUR_SIX_TIE_BLOCK
    bits = (row.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), row)  # exact in bf16
    return bits


def test_four_six_tie_keeps_the_six_candidate(O):
    f = np.float32
    x = four_six_tie_row()[None, :]
    c46, s46, t = O.nvfp4_quantize_rows(x, four_six=True)
    assert t[0] == f(50.75) / f(2688)
    d6, d4 = f(256.0) * t[0], f(384.0) * t[0]        # E4M3 0x78 = 256, 0x7C = 384
    # the outlier's reconstruction and error, binary32 step by step
    assert f(6.0) * d6 == f(29.0) and f(4.0) * d4 == f(29.0)
    assert np.float64(6.0) * np.float64(d6) != 29.0    # exact product: not a tie
    blk = np.array(FOUR_SIX_TIE_BLOCK, np.float32)
    cc6, ss6, sse6 = O.nvfp4_block_candidate(blk, t[0], 6.0)
    cc4, ss4, sse4 = O.nvfp4_block_candidate(blk, t[0], 4.0)
    assert (ss6, ss4) == (0x78, 0x7C)
    assert sse6 == sse4
    assert s46[0, 1] == 0x78
    assert np.array_equal(unpack(c46[:, 8:16])[0], cc6)


def test_mxfp8_against_torch_float8(O):
    x = synth.rows_log_uniform_std(64, 256, seed=2)
    rc, rs, cc, cs = O.mxfp8_quantize_rowcol(x)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    blocks = xf.reshape(64, 8, 32)
    amax = np.abs(blocks).max(axis=2)
    _, e = np.frexp(amax)                          # amax = m * 2^e, m in [0.5, 1)
    X = np.clip((e - 1) - 8, -127, 127)
    assert np.array_equal(rs.astype(np.int64), X + 127)
    y = np.clip(blocks * np.exp2(-X)[:, :, None], -448, 448).astype(np.float32)
    ref = torch.from_numpy(y.reshape(64, 256)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(rc, ref)
    # the scaled block maximum lands in [256, 512)
    top = np.abs(blocks).max(axis=2) * np.exp2(-X)
    assert np.all((top >= 256) & (top < 512))


def test_mxfp8_column_copy_is_row_copy_of_transpose(O):
    x = synth.rows_log_uniform_std(96, 160, seed=3)
    rc, rs, cc, cs = O.mxfp8_quantize_rowcol(x)
    xt = np.ascontiguousarray(x.T)
    trc, trs, _, _ = O.mxfp8_quantize_rowcol(xt, col=False)
    assert np.array_equal(cc, trc) and np.array_equal(cs, trs)
    # both copies come from the original bf16 (the row copy alone gives the same bytes)
    rc2, rs2, _, _ = O.mxfp8_quantize_rowcol(x, col=False)
    assert np.array_equal(rc, rc2) and np.array_equal(rs, rs2)


def test_mxfp8_zero_block(O):
    x = np.zeros((32, 64), np.uint16)
    x[3, 40] = synth.to_bf16_bits(np.array([3.0], np.float32))[0]
    rc, rs, cc, cs = O.mxfp8_quantize_rowcol(x)
    assert rs[0, 0] == 0 and not rc[0].any()
    assert rs[3, 1] == 1 - 8 + 127 and cs[40, 0] == 1 - 8 + 127
    assert not cc[0].any() and cs[0, 0] == 0


def _identity_requant_input(M, K, seed):
    """NVFP4 input with t = 1 and block scale 1 whose values are E2M1 grid
    points and whose every 16-run down a column has an element of
    magnitude 6, so requantization must reproduce the codes transposed."""
    g = np.random.default_rng(seed)
    codes_u = g.integers(0, 16, size=(M, K)).astype(np.uint8)
    r = g.integers(0, 16, size=(M // 16, K))
    for b in range(M // 16):
        codes_u[16 * b + r[b], np.arange(K)] = g.choice([0x7, 0xF], size=K)
    packed = (codes_u[:, 0::2] | (codes_u[:, 1::2] << 4)).astype(np.uint8)
    sf = np.full((M, K // 16), 0x38, np.uint8)     # E4M3 1.0
    return codes_u, packed, sf, np.ones(M, np.float32)


def test_requant_rne_identity_up_to_transpose(O):
    M, K = 96, 64
    codes_u, packed, sf, t = _identity_requant_input(M, K, seed=1)
    nc, ns, nt, mc, ms = O.requant_transpose(packed, sf, t, sr=False, seed=0)
    assert np.array_equal(unpack(nc), codes_u.T)
    assert np.all(ns == 0x7E)                       # every block scale 448
    assert np.all(nt == np.float32(6.0) / np.float32(2688.0))
    # MXFP8 target: amax 6 -> X = 2 - 8 = -6, codes = E4M3(value * 64)
    assert np.all(ms == 121)
    vals = e2m1_val(codes_u.T) * 64.0
    ref = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mc, ref)
    # SR never moves values that are already on the grid
    nc2, ns2, nt2, mc2, ms2 = O.requant_transpose(packed, sf, t, sr=True, seed=123)
    assert np.array_equal(nc2, nc) and np.array_equal(mc2, mc)


def test_requant_matches_quantizing_the_dequantized_transpose(O):
    x = synth.normal_with_outliers(64, 96, seed=7)
    codes, sf, t = O.nvfp4_quantize_rows(x)
    nc, ns, nt, mc, ms = O.requant_transpose(codes, sf, t, sr=False, seed=0)
    D = O.nvfp4_dequantize(codes, sf, t)
    # bf16-representable? not in general; compare through the binary32 path
    c2, s2 = O.nvfp4_quantize_rows_given_t(D.T.copy(), nt)
    assert np.array_equal(nc, c2) and np.array_equal(ns, s2)
    assert np.array_equal(nt, (np.abs(D).max(axis=0) / np.float32(2688)).astype(np.float32))


def test_sr_draws_depend_only_on_output_index(O):
    x = synth.normal_with_outliers(64, 64, seed=8)
    codes, sf, t = O.nvfp4_quantize_rows(x)
    a = O.requant_transpose(codes, sf, t, sr=True, seed=7)
    b = O.requant_transpose(codes, sf, t, sr=True, seed=7)
    c = O.requant_transpose(codes, sf, t, sr=True, seed=8)
    for i in (0, 3):
        assert np.array_equal(a[i], b[i])
    assert not np.array_equal(a[0], c[0])
    assert np.array_equal(a[1], c[1]) and np.array_equal(a[2], c[2])  # scales are RNE


# ---------------------------------------------------------------- dequantize to bf16
def _bf16_bits_of_exact(v):
    """bf16 bits of a value that bf16 holds exactly (pure Python packing)."""
    import struct
    b = struct.unpack("<I", struct.pack("<f", v))[0]
    assert b & 0xFFFF == 0, v
    return b >> 16


def test_dequant_bf16_exact_products(O):
    # every code under block scales across the E4M3 range (0x01 = 2^-9 up to
    # 0x7E = 448) and power-of-two row scales: each product has at most 5
    # significant bits, so the bf16 result is the exact value; -0 keeps its sign
    nib = np.arange(16, dtype=np.uint8)
    packed = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)
    sfs = [0x01, 0x08, 0x30, 0x38, 0x3F, 0x7E]
    codes = np.tile(packed, (len(sfs), 1))
    sf = np.array(sfs, np.uint8).reshape(-1, 1)
    for t in (1.0, 2.0 ** -7, 2.0 ** 20):
        out = O.nvfp4_dequantize_bf16(codes, sf, np.full(len(sfs), t, np.float32))
        for i, s in enumerate(sfs):
            for k in range(16):
                v = float(e2m1_val(k)) * float(e4m3_val(s)) * t
                assert out[i, k] == _bf16_bits_of_exact(v), (hex(s), k, t)


def test_dequant_bf16_rounding_against_numpy_and_torch(O):
    # arbitrary row scales: binary32 products from numpy's float32 arithmetic,
    # then torch's round-to-nearest-even conversion to bf16
    codes, sf, t = synth.random_nvfp4(64, 256, seed=11)
    out = O.nvfp4_dequantize_bf16(codes, sf, t)
    v = e2m1_val(unpack(codes)).astype(np.float32)
    s = np.repeat(e4m3_val(sf).astype(np.float32), 16, axis=1)
    f32 = (v * s) * t[:, None]
    ref = torch.from_numpy(np.ascontiguousarray(f32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(out, ref)


def test_dequant_bf16_ties_to_even(O):
    # 1.0 * (1 + 2^-8) is halfway between bf16 1.0 (0x3F80) and 1 + 2^-7
    # (0x3F81): the even one, 0x3F80.  1 + 3 * 2^-8 is halfway between 0x3F81
    # and 0x3F82: 0x3F82.
    codes = np.full((1, 8), 0x22, np.uint8)  # code 2 (= 1.0) in both nibbles
    sf = np.array([[0x38]], np.uint8)        # E4M3 1.0
    assert (O.nvfp4_dequantize_bf16(codes, sf, np.array([1 + 2.0 ** -8], np.float32)) == 0x3F80).all()
    assert (O.nvfp4_dequantize_bf16(codes, sf, np.array([1 + 3 * 2.0 ** -8], np.float32)) == 0x3F82).all()


# ---------------------------------------------------------------- 2-D (16 x 16) block scales
def _transpose_codes(codes):
    """Packed [rows, K/2] -> the packed codes of the transpose, [K, rows/2]."""
    u = unpack(codes).T
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def test_2d_transpose_invariance(O):
    # the tile maxima and the per-tensor scale do not change under the
    # transpose and the element rule is elementwise, so quantizing x^T gives
    # the transposed codes and tile scales
    x = synth.normal_with_outliers(64, 96, seed=21)
    c, s, t = O.nvfp4_quantize_2d(x)
    cT, sT, tT = O.nvfp4_quantize_2d(np.ascontiguousarray(x.T))
    assert t == tT
    np.testing.assert_array_equal(cT, _transpose_codes(c))
    np.testing.assert_array_equal(sT, s.T)


def test_2d_uniform_tile_closed_form(O):
    # x = 1 everywhere: t = 1/2688, tile scale E4M3(1 / (6 t)) = 448 (0x7E),
    # d = 448 t = 1/6, so every element becomes 6 (code 7)
    x = np.full((16, 32), 0x3F80, np.uint16)
    c, s, t = O.nvfp4_quantize_2d(x)
    assert np.float32(t) == np.float32(1.0) / np.float32(2688.0)
    assert (s == 0x7E).all()
    assert (unpack(c) == 7).all()


def test_2d_reduces_to_per_row_for_repeated_rows(O):
    # identical rows: each tile's maximum is its 16-blocks' maximum and the
    # per-tensor scale is every row's scale, so the result is the 1 x 16 one
    row = synth.normal_with_outliers(1, 64, seed=22)
    x = np.repeat(row, 32, axis=0)
    c2, s2, t2 = O.nvfp4_quantize_2d(x)
    c1, s1, t1 = O.nvfp4_quantize_rows(x)
    assert (np.asarray(t1, np.float32) == np.float32(t2)).all()
    np.testing.assert_array_equal(c2, c1)
    np.testing.assert_array_equal(np.repeat(s2, 16, axis=0), s1)


def test_2d_one_outlier_flushes_its_tile(O):
    # the page's objection to square blocks: one large value among 256 pushes
    # the other 255 to zero, while with 1 x 16 blocks only the outlier's own
    # block loses its small values
    x = np.full((16, 16), 0x3F80, np.uint16)  # 1.0
    x[5, 9] = 0x447A                          # 1000.0
    u2 = unpack(O.nvfp4_quantize_2d(x)[0])
    assert u2[5, 9] == 7
    assert (np.delete(u2.ravel(), 5 * 16 + 9) == 0).all()
    u1 = unpack(O.nvfp4_quantize_rows(x)[0])
    assert (u1[np.arange(16) != 5] == 7).all()
    assert u1[5, 9] == 7 and (np.delete(u1[5], 9) == 0).all()


def test_2d_zero_tensor(O):
    c, s, t = O.nvfp4_quantize_2d(np.zeros((32, 48), np.uint16))
    assert t == 0.0 and not c.any() and not s.any()


# ---------------------------------------------------------------- 32-point random Hadamard transform
def _hadamard32():
    import scipy.linalg
    return scipy.linalg.hadamard(32).astype(np.float64)  # Sylvester construction


def test_rht_unit_vectors_give_hadamard_columns(O):
    H = _hadamard32()
    signs = O.rht_signs(7)
    s = np.where((signs >> np.arange(32)) & 1, -1.0, 1.0)
    for k in range(32):
        e = np.zeros(32, np.float32)
        e[k] = 1.0
        np.testing.assert_array_equal(O.rht32(e, 0), H[:, k])
        np.testing.assert_array_equal(O.rht32(e, signs), s[k] * H[:, k])


def test_rht_exact_on_small_integers_and_inverts(O):
    # integer inputs up to 8 keep every butterfly sum exact in binary32, so the
    # transform equals H (s . x) in float64, and H H = 32 I undoes it
    rng = np.random.default_rng(3)
    x = rng.integers(-8, 9, size=(4, 96)).astype(np.float32)
    signs = O.rht_signs(11)
    s = np.where((signs >> np.arange(32)) & 1, -1.0, 1.0)
    y = O.rht32(x, signs)
    ref = (x.reshape(-1, 32).astype(np.float64) * s) @ _hadamard32().T
    np.testing.assert_array_equal(y.reshape(-1, 32), ref)
    back = O.rht32(y, 0).reshape(-1, 32) * s / 32.0
    np.testing.assert_array_equal(back.reshape(x.shape), x)


def test_rht_binary32_rounding_bound(O):
    # arbitrary values: five binary32 additions per output, so each output is
    # within 5 * 2^-24 * sum|x| of the exact transform
    x = synth.bf16_bits_to_f32(synth.normal_with_outliers(8, 256, seed=4)).astype(np.float32)
    signs = O.rht_signs(5)
    s = np.where((signs >> np.arange(32)) & 1, -1.0, 1.0)
    y = O.rht32(x, signs).reshape(-1, 32).astype(np.float64)
    g = x.reshape(-1, 32).astype(np.float64)
    exact = (g * s) @ _hadamard32().T
    bound = 5 * 2.0 ** -24 * np.abs(g).sum(axis=1, keepdims=True)
    assert (np.abs(y - exact) <= bound).all()


def test_rht_quantization_is_the_per_row_recipe_of_the_transform(O):
    x = synth.normal_with_outliers(16, 128, seed=6)
    c, s, t = O.nvfp4_quantize_rht(x, seed=9)
    y = O.rht32(synth.bf16_bits_to_f32(x).astype(np.float32), O.rht_signs(9))
    t_ref = (np.abs(y).max(axis=1) / np.float32(2688.0)).astype(np.float32)
    np.testing.assert_array_equal(t, t_ref)
    c2, s2 = O.nvfp4_quantize_rows_given_t(y, t_ref)
    np.testing.assert_array_equal(c, c2)
    np.testing.assert_array_equal(s, s2)


def _nearest_e2m1_code(v):
    """Brute-force E2M1 encoder, independent of the oracle's table: the
    nearest of the 8 magnitudes by exact fp64 distance, ties to the even code,
    saturating at 6, the sign bit taken from the input (so -0.0 -> 0x8)."""
    v = np.asarray(v, np.float32)
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    a = np.abs(v.astype(np.float64))
    dist = np.abs(a[..., None] - mags)
    best = dist.min(axis=-1, keepdims=True)
    ties = dist == best
    # among the tied magnitudes prefer an even code index (0, 2, 4, 6)
    even = ties & (np.arange(8) % 2 == 0)
    idx = np.where(even.any(axis=-1), even.argmax(axis=-1), ties.argmax(axis=-1))
    idx = np.where(a >= 6.0, 7, idx)
    return (idx | (np.signbit(v).astype(np.int64) << 3)).astype(np.uint8)


def _e4m3_rne(v):
    """binary32 -> E4M3 byte by torch's float8_e4m3fn conversion (round to
    nearest even), independent of the oracle's encoder."""
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_block_scale_and_codes_at_general_t(O):
    """Steps 3 and 4 of the per-token recipe at per-token scales t != 1, each
    byte recomputed with encoders that share nothing with the oracle: the
    block scale is E4M3(rn(amax_b / rn(6 t))) by torch's float8 conversion,
    the code the nearest E2M1 of rn(x * rn(1 / d)) with d = rn(E4M3(sf) * t),
    by brute force ("End-to-End 4-Bit Training", section "先说为什么难": 16
    E2M1 values share an E4M3 scale, and a second FP32 scale per token)."""
    x = np.concatenate([synth.normal_with_outliers(192, 512, seed=41),
                        synth.rows_log_uniform_std(64, 512, seed=42, lo_exp=-20, hi_exp=20)])
    codes, sf, t = O.nvfp4_quantize_rows(x)
    assert np.any(t != np.float32(1.0))
    xf = synth.bf16_bits_to_f32(x).astype(np.float32)
    rows, K = xf.shape
    blocks = xf.reshape(rows, K // 16, 16)
    amax_b = np.abs(blocks).max(axis=-1).astype(np.float32)
    six_t = (np.float32(6.0) * t).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        s_raw = np.where(six_t[:, None] > 0, amax_b / six_t[:, None], np.float32(0)).astype(np.float32)
    assert np.array_equal(sf, _e4m3_rne(s_raw)), "block scale bytes"
    d = (e4m3_val(sf).astype(np.float32) * t[:, None]).astype(np.float32)   # exact product, one rounding
    with np.errstate(divide="ignore", over="ignore"):
        enc = np.where(d > 0, np.float32(1.0) / d, np.float32(0)).astype(np.float32)
    enc = np.where(np.isinf(enc), np.finfo(np.float32).max, enc).astype(np.float32)
    y = (blocks * enc[..., None]).astype(np.float32)
    want = _nearest_e2m1_code(y).reshape(rows, K)
    assert np.array_equal(unpack(codes), want), "element codes"
    # the check has power against a division in place of the reciprocal:
    # x / d differs from rn(x * rn(1/d)) on enough of these elements to flip codes
    with np.errstate(divide="ignore", invalid="ignore"):
        y_div = np.where(d[..., None] > 0, blocks / d[..., None], np.float32(0)).astype(np.float32)
    assert not np.array_equal(_nearest_e2m1_code(y_div).reshape(rows, K), want)


def test_block_scale_at_general_t_detects_an_extra_rounding(O):
    """The same block-scale pin has power against rounding 6 t twice (or
    dividing by 6 then by t): on these rows at least one scale byte differs."""
    x = synth.normal_with_outliers(256, 512, seed=43)
    _, sf, t = O.nvfp4_quantize_rows(x)
    xf = synth.bf16_bits_to_f32(x).astype(np.float32)
    amax_b = np.abs(xf.reshape(256, 32, 16)).max(axis=-1).astype(np.float32)
    two_step = ((amax_b / np.float32(6.0)).astype(np.float32) / t[:, None]).astype(np.float32)
    assert not np.array_equal(sf, _e4m3_rne(two_step))
