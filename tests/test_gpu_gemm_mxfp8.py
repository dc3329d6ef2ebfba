"""GPU: the grouped GEMM on MXFP8 operands (tcgen05.mma kind::mxf8f6f4, one
E8M0 scale per 32 elements) against the oracle's fp64 GEMM on exactly
dequantized operands, with the NVFP4 GEMM's tolerances: relative Frobenius
error <= 1e-5 and per-element |err| <= 1e-4 * sum_k |a_k b_k| (fp32 outputs);
bf16 outputs add half a bf16 ulp.  Includes the weight-gradient GEMM fed by
the column copies of the MXFP8 quantizer."""
import numpy as np
import pytest
import torch

from block_scaled_precision_quantize_gb300 import synth
from conftest import to_dev, to_np

pytestmark = pytest.mark.gpu

REL_FRO = 1e-5
REL_ABS = 1e-4


def _problem(O, counts, K, N, seed):
    E = len(counts)
    pads = [(c + 127) // 128 * 128 for c in counts]
    offsets = np.concatenate([[0], np.cumsum(pads)]).astype(np.int32)
    M = int(offsets[-1])
    x = synth.rows_log_uniform_std(M, K, seed=seed)
    ac, asf, _, _ = O.mxfp8_quantize_rowcol(x, col=False)
    for e in range(E):
        ac[offsets[e] + counts[e]:offsets[e + 1]] = 0  # padding rows: zero codes
    w = synth.normal((E * N, K), seed=seed + 1, std=0.02)
    bc, bsf, _, _ = O.mxfp8_quantize_rowcol(w, col=False)
    return offsets, M, ac, asf, bc, bsf


def _reference(O, offsets, ac, asf, bc, bsf, E, N):
    M = ac.shape[0]
    ref, ab = np.zeros((M, N)), np.zeros((M, N))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            o, a = O.gemm_mxfp8(ac[r0:r1], asf[r0:r1], np.ones(r1 - r0, np.float32), bc[e * N:(e + 1) * N],
                                bsf[e * N:(e + 1) * N], 1.0)
            ref[r0:r1], ab[r0:r1] = o, a
    return ref, ab


def _run(gpu, O, offsets, ac, asf, bc, bsf, E, N, epilogue):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu.grouped_expert_gemm_mxfp8(to_dev(ac), to_dev(O.sf_to_swizzled(asf)), to_dev(offsets),
                                        to_dev(bc.reshape(E, N, -1)), to_dev(O.sf_to_swizzled(bsf)),
                                        epilogue=epilogue, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return to_np(out).astype(np.float64) if epilogue == gpu.EPI_F32 else \
        torch.from_numpy(to_np(out).view(np.int16)).view(torch.bfloat16).double().numpy()


def _assert_close(got, ref, ab, extra=0.0):
    err = np.abs(got - ref)
    bad = np.argwhere(err > REL_ABS * ab + extra * np.abs(ref) + 1e-30)
    assert bad.size == 0, f"{bad.shape[0]} out of bound; first {tuple(bad[0])}: got {got[tuple(bad[0])]} " \
                          f"ref {ref[tuple(bad[0])]}"
    if extra == 0.0:
        assert np.linalg.norm(got - ref) <= REL_FRO * max(np.linalg.norm(ref), 1e-300)


def test_mxfp8_gemm_integer_exact_single_tile(gpu, O):
    # E4M3 codes of small integers with unit block scales: exact fp32 sums
    rng = np.random.default_rng(1)
    vals = np.array([0x00, 0x38, 0x40, 0x44, 0xC0], np.uint8)
    ints = np.array([0, 1, 2, 3, -2], np.float64)
    ia, ib = rng.integers(0, 5, size=(128, 256)), rng.integers(0, 5, size=(128, 256))
    sa, sb = np.full((128, 8), 127, np.uint8), np.full((128, 8), 127, np.uint8)
    got = _run(gpu, O, np.array([0, 128], np.int32), vals[ia], sa, vals[ib], sb, 1, 128, gpu.EPI_F32)
    np.testing.assert_array_equal(got, ints[ia] @ ints[ib].T)


@pytest.mark.parametrize("counts,K,N", [([128], 128, 128), ([200, 0, 77], 256, 384), ([300, 129], 768, 256)])
@pytest.mark.parametrize("bf16", [False, True])
def test_mxfp8_gemm_matches_oracle(gpu, O, counts, K, N, bf16):
    offsets, M, ac, asf, bc, bsf = _problem(O, counts, K, N, seed=len(counts) + K)
    E = len(counts)
    got = _run(gpu, O, offsets, ac, asf, bc, bsf, E, N, gpu.EPI_BF16 if bf16 else gpu.EPI_F32)
    ref, ab = _reference(O, offsets, ac, asf, bc, bsf, E, N)
    _assert_close(got, ref, ab, extra=2.0 ** -8 if bf16 else 0.0)


def test_mxfp8_weight_gradient_from_column_copies(gpu, O):
    # dW[n][k] = sum_t dY[t][n] X[t][k]: both operands are the column copies
    # (stored transposed, blocks of 32 along t) that the MXFP8 quantizer emits
    # for the backward pass, with K = T tokens
    T, Nout, Kin = 512, 256, 384
    dy = synth.normal_with_outliers(T, Nout, seed=11)
    x = synth.normal_with_outliers(T, Kin, seed=12)
    dyq = gpu.quantize_mxfp8_rowcol(to_dev(dy), row=False, swizzled=True)
    xq = gpu.quantize_mxfp8_rowcol(to_dev(x), row=False, swizzled=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu.grouped_expert_gemm_mxfp8(dyq[2], dyq[3], torch.tensor([0, Nout], dtype=torch.int32, device="cuda"),
                                        xq[2].reshape(1, Kin, T), xq[3], dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _, _, dcc, dcs = O.mxfp8_quantize_rowcol(dy, row=False)
    _, _, xcc, xcs = O.mxfp8_quantize_rowcol(x, row=False)
    assert np.array_equal(to_np(dyq[2]), dcc) and np.array_equal(to_np(xq[2]), xcc)
    ref, ab = O.gemm_mxfp8(dcc, dcs, np.ones(Nout, np.float32), xcc, xcs, 1.0)
    _assert_close(to_np(out).astype(np.float64), ref, ab)
