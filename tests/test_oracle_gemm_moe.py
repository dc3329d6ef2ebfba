"""Oracle pins for the block-scaled GEMM, routing, SwiGLU and combine (CPU):
brute force against numpy's fp64 matmul on independently decoded operands,
an integer-exact special case, stable-sort routing and closed forms."""
import math

import numpy as np
import torch

from block_scaled_precision_quantize_gb300 import synth

E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])


def _deq64(codes, sf, t):
    """Independent fp64 decode: E2M1 from the value list, E4M3 via torch."""
    c = np.asarray(codes, np.uint8)
    u = np.empty(c.shape[:-1] + (c.shape[-1] * 2,), np.int64)
    u[..., 0::2] = c & 0xF
    u[..., 1::2] = c >> 4
    s = torch.from_numpy(np.ascontiguousarray(sf)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return E2M1[u] * np.repeat(s, 16, axis=-1) * np.asarray(t, np.float64)[..., None]


def test_gemm_matches_numpy_fp64(O):
    a = synth.normal_with_outliers(40, 320, seed=1)
    w = synth.normal((1, 72, 320), seed=2, std=0.02)
    ac, asf, at = O.nvfp4_quantize_rows(a)
    wc, wsf, wt = O.nvfp4_quantize_group(w)
    out, ab = O.gemm_nvfp4(ac, asf, at, wc[0], wsf[0], wt[0])
    A = _deq64(ac, asf, at)
    B = _deq64(wc[0], wsf[0], np.full(72, wt[0]))
    ref = A @ B.T
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-14 * np.abs(A).max() * np.abs(B).max())
    assert np.allclose(ab, np.abs(A) @ np.abs(B).T, rtol=1e-12)


def test_gemm_integer_exact_case(O):
    # block scales 1 and FP32 scales 1: every product is a multiple of 0.25
    # and the sum is exact, so the result equals an integer matmul / 4
    g = np.random.default_rng(5)
    M, N, K = 24, 40, 256
    au = g.integers(0, 16, (M, K))
    bu = g.integers(0, 16, (N, K))
    pack = lambda u: (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)
    one = np.full((M, K // 16), 0x38, np.uint8)
    out, _ = O.gemm_nvfp4(pack(au), one, np.ones(M, np.float32), pack(bu),
                          np.full((N, K // 16), 0x38, np.uint8), 1.0)
    ai = (E2M1[au] * 2).astype(np.int64)
    bi = (E2M1[bu] * 2).astype(np.int64)
    assert np.array_equal(out * 4, (ai @ bi.T).astype(np.float64))


def test_gemm_sampled_equals_full(O):
    a = synth.normal_with_outliers(32, 256, seed=3)
    w = synth.normal((2, 64, 256), seed=4, std=0.02)
    ac, asf, at = O.nvfp4_quantize_rows(a)
    wc, wsf, wt = O.nvfp4_quantize_group(w)
    full1, _ = O.gemm_nvfp4(ac, asf, at, wc[1], wsf[1], wt[1])
    rows = np.array([0, 5, 31, 7])
    cols = np.array([3, 63, 0, 17])
    s, sab = O.gemm_nvfp4_sampled(ac, asf, at, wc.reshape(128, -1), wsf.reshape(128, -1), wt,
                                  rows, cols + 64, np.ones(4, np.int64))
    assert np.array_equal(s, full1[rows, cols])


def test_route_is_a_stable_sort_by_expert(O):
    T, k, E = 300, 4, 7
    g = np.random.default_rng(0)
    ids = np.stack([g.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    ids[:, 0] = np.where(np.arange(T) % 5 == 0, 3, ids[:, 0])  # skew
    offsets, slot_of, row_src = O.route(ids, E, pad=128)
    flat = ids.ravel()
    order = sorted(range(T * k), key=lambda i: (flat[i], i))
    counts = np.bincount(flat, minlength=E)
    pads = (counts + 127) // 128 * 128
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(pads)]).astype(np.int32))
    pos = {}
    for e in range(E):
        mine = [i for i in order if flat[i] == e]
        for j, i in enumerate(mine):
            pos[i] = offsets[e] + j
    assert all(slot_of[i] == pos[i] for i in range(T * k))
    assert row_src.size == offsets[-1]
    assert np.all(row_src[slot_of] == np.arange(T * k))
    assert (row_src == -1).sum() == offsets[-1] - T * k


def test_swiglu_closed_forms(O):
    g = np.array([0.0, 1.0, -1.0, 30.0, -30.0, 2.5])
    u = np.array([3.0, 2.0, 2.0, 1.0, 1.0, -4.0])
    h = O.swiglu(np.concatenate([g, u])[None, :])[0]
    ref = [0.0, 2.0 / (1 + math.exp(-1)), -2.0 / (1 + math.e), 30.0 / (1 + math.exp(-30)),
           -30.0 / (1 + math.exp(30)), -4.0 * 2.5 / (1 + math.exp(-2.5))]
    assert np.allclose(h, ref, rtol=1e-15, atol=1e-300)
    assert h[0] == 0.0 and abs(h[3] - 30.0) < 1e-11 and abs(h[4]) < 1e-11


def test_combine_closed_forms(O):
    T, k, H = 5, 3, 8
    g = np.random.default_rng(1)
    out = synth.to_bf16_bits(g.standard_normal((T * k + 4, H)).astype(np.float32))
    slot_of = g.permutation(T * k + 4)[:T * k].astype(np.int32)
    w = np.zeros((T, k), np.float32)
    w[:, 1] = 1.0                                   # one-hot: y is that row
    y = O.combine(out, slot_of, w)
    assert np.array_equal(y, out[slot_of.reshape(T, k)[:, 1]])
    w = np.full((T, k), 0.5, np.float32)            # 0.5 * (a + b + c), exact in fp64
    y = O.combine(out, slot_of, w)
    of = synth.bf16_bits_to_f32(out).astype(np.float64)
    ref = 0.5 * of[slot_of.reshape(T, k)].sum(axis=1)
    yf = synth.bf16_bits_to_f32(y).astype(np.float64)
    assert np.all(np.abs(yf - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-38)


# ---------------------------------------------------------------- MXFP8 GEMM (the backward's operands)
def _mx_deq64(codes, sf):
    """Independent fp64 decode of MXFP8: E4M3 via torch, E8M0 as 2^(b - 127)."""
    c = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    s = np.exp2(np.asarray(sf, np.float64) - 127.0)
    return c * np.repeat(s, 32, axis=-1)


def test_mxfp8_gemm_matches_numpy_fp64(O):
    a = synth.rows_log_uniform_std(64, 256, seed=3)
    w = synth.normal((48, 256), seed=4, std=0.02)
    ac, asf, _, _ = O.mxfp8_quantize_rowcol(a, col=False)
    wc, wsf, _, _ = O.mxfp8_quantize_rowcol(w, col=False)
    ones = np.ones(64, np.float32)
    out, ab = O.gemm_mxfp8(ac, asf, ones, wc, wsf, 1.0)
    A, B = _mx_deq64(ac, asf), _mx_deq64(wc, wsf)
    ref = A @ B.T
    assert np.all(np.abs(out - ref) <= 1e-12 * (np.abs(A) @ np.abs(B).T) + 1e-300)
    np.testing.assert_allclose(ab, np.abs(A) @ np.abs(B).T, rtol=1e-12)


def test_mxfp8_gemm_integer_exact_case(O):
    # E4M3 codes of small integers (0x38 = 1, 0x40 = 2, 0x44 = 3, 0xC0 = -2) and
    # unit block scales (E8M0 127): the sums are exact integers
    rng = np.random.default_rng(5)
    vals = np.array([0x00, 0x38, 0x40, 0x44, 0xC0], np.uint8)
    ints = np.array([0, 1, 2, 3, -2], np.float64)
    ia = rng.integers(0, 5, size=(16, 64))
    ib = rng.integers(0, 5, size=(8, 64))
    sa = np.full((16, 2), 127, np.uint8)
    sb = np.full((8, 2), 127, np.uint8)
    out, _ = O.gemm_mxfp8(vals[ia], sa, np.ones(16, np.float32), vals[ib], sb, 1.0)
    np.testing.assert_array_equal(out, ints[ia] @ ints[ib].T)
    # block scale 2^1 on A's second block of 32 doubles exactly that half's share
    sa[:, 1] = 128
    out2, _ = O.gemm_mxfp8(vals[ia], sa, np.ones(16, np.float32), vals[ib], sb, 1.0)
    np.testing.assert_array_equal(out2, ints[ia][:, :32] @ ints[ib][:, :32].T + 2 * ints[ia][:, 32:] @ ints[ib][:, 32:].T)
