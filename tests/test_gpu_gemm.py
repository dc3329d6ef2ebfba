"""GPU: the tcgen05 block-scaled grouped GEMM against the oracle's fp64 GEMM
on exactly dequantized operands.  Tolerances: relative Frobenius error
<= 1e-5 and per-element |err| <= 1e-4 * sum_k |a_k b_k| (fp32 outputs); bf16
outputs add half a bf16 ulp of the value."""
import numpy as np
import pytest
import torch

from block_scaled_precision_quantize_gb300 import synth
from conftest import to_dev, to_np

pytestmark = pytest.mark.gpu

REL_FRO = 1e-5
REL_ABS = 1e-4


def _pack(u):
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def _make_problem(O, counts, K, N, seed):
    """Expert-sorted A (segments padded to 128 rows; padding rows are zero
    codes with zero scale) and per-expert B, quantized by the oracle."""
    E = len(counts)
    pads = [(c + 127) // 128 * 128 for c in counts]
    offsets = np.concatenate([[0], np.cumsum(pads)]).astype(np.int32)
    M = int(offsets[-1])
    x = synth.normal_with_outliers(max(M, 1), K, seed=seed)
    ac, asf, at = O.nvfp4_quantize_rows(x)
    for e in range(E):
        pad0 = offsets[e] + counts[e]
        ac[pad0:offsets[e + 1]] = 0
        asf[pad0:offsets[e + 1]] = 0
        at[pad0:offsets[e + 1]] = 0
    w = synth.normal((E, N, K), seed=seed + 1, std=0.02)
    bc, bsf, bt = O.nvfp4_quantize_group(w)
    return offsets, M, (ac, asf, at), (bc, bsf, bt)


def _reference(O, offsets, A, B):
    ac, asf, at = A
    bc, bsf, bt = B
    E, N = bc.shape[0], bc.shape[1]
    M = ac.shape[0]
    ref = np.zeros((M, N))
    ab = np.zeros((M, N))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            o, a = O.gemm_nvfp4(ac[r0:r1], asf[r0:r1], at[r0:r1], bc[e], bsf[e], bt[e])
            ref[r0:r1], ab[r0:r1] = o, a
    return ref, ab


def _run(gpu, O, offsets, A, B, epilogue):
    ac, asf, at = A
    bc, bsf, bt = B
    E, N, Kh = bc.shape
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu.grouped_expert_gemm_fp4(to_dev(ac), to_dev(O.sf_to_swizzled(asf)), to_dev(at), to_dev(offsets),
                                      to_dev(bc), to_dev(O.sf_to_swizzled(bsf.reshape(E * N, -1))), to_dev(bt),
                                      epilogue=epilogue, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out


def _assert_close(got, ref, ab, extra=0.0):
    err = np.abs(got.astype(np.float64) - ref)
    fro = np.linalg.norm(got.astype(np.float64) - ref) / max(np.linalg.norm(ref), 1e-300)
    bound = REL_ABS * ab + extra * np.abs(ref) + 1e-30
    bad = np.argwhere(err > bound)
    assert bad.size == 0, f"{bad.shape[0]} elements out of bound; first {tuple(bad[0])}: got " \
                          f"{got[tuple(bad[0])]} ref {ref[tuple(bad[0])]}"
    if extra == 0.0:
        assert fro <= REL_FRO, fro


def test_gemm_integer_exact_single_tile(gpu, O):
    """Block scales 1 and FP32 scales 1: the result is an exact integer
    matmul / 4, so any layout, swizzle or descriptor error shows."""
    g = np.random.default_rng(1)
    M, N, K = 128, 128, 256
    au = g.integers(0, 16, (M, K))
    bu = g.integers(0, 16, (N, K))
    ac, bc = _pack(au), _pack(bu)
    asf = np.full((M, K // 16), 0x38, np.uint8)
    bsf = np.full((N, K // 16), 0x38, np.uint8)
    one_a, one_b = np.ones(M, np.float32), np.ones(1, np.float32)
    out = gpu.grouped_expert_gemm_fp4(to_dev(ac), to_dev(O.sf_to_swizzled(asf)), to_dev(one_a),
                                      to_dev(np.array([0, M], np.int32)), to_dev(bc[None]),
                                      to_dev(O.sf_to_swizzled(bsf)), to_dev(one_b))
    ref, _ = O.gemm_nvfp4(ac, asf, one_a, bc, bsf, 1.0)
    got = to_np(out).astype(np.float64)
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:5]


def test_gemm_scaled_single_tile(gpu, O):
    offsets, M, A, B = _make_problem(O, [128], 256, 128, seed=2)
    out = _run(gpu, O, offsets, A, B, gpu.EPI_F32)
    ref, ab = _reference(O, offsets, A, B)
    _assert_close(to_np(out), ref, ab)


@pytest.mark.parametrize("counts,K,N", [([128], 2048, 256), ([100, 0, 300], 576, 384), ([1, 129, 64, 7], 256, 512),
                                        ([513], 1024, 128)])
def test_gemm_grouped_f32(gpu, O, counts, K, N):
    offsets, M, A, B = _make_problem(O, counts, K, N, seed=sum(counts) + K)
    out = _run(gpu, O, offsets, A, B, gpu.EPI_F32)
    ref, ab = _reference(O, offsets, A, B)
    _assert_close(to_np(out), ref, ab)


def test_gemm_bf16_epilogue(gpu, O):
    offsets, M, A, B = _make_problem(O, [200, 56], 512, 256, seed=9)
    out = _run(gpu, O, offsets, A, B, gpu.EPI_BF16)
    ref, ab = _reference(O, offsets, A, B)
    got = synth.bf16_bits_to_f32(to_np(out))
    _assert_close(got, ref, ab, extra=2.0 ** -8)


def test_gemm_swiglu_epilogue(gpu, O):
    counts, K, I = [150, 90], 512, 256
    offsets, M, A, B = _make_problem(O, counts, K, 2 * I, seed=12)
    out = _run(gpu, O, offsets, A, B, gpu.EPI_SWIGLU_BF16)
    ref, ab = _reference(O, offsets, A, B)
    h = O.swiglu(ref)
    # error propagation: |dh| <= |silu'(g)| |u| |dg| + |silu(g)| |du|, silu' <= 1.1
    g, u = ref[:, :I], ref[:, I:]
    dg, du = REL_ABS * ab[:, :I], REL_ABS * ab[:, I:]
    sg = g / (1 + np.exp(-g))
    bound = 1.1 * np.abs(u) * dg + np.abs(sg) * du + 2.0 ** -8 * np.abs(h) + 1e-30
    got = synth.bf16_bits_to_f32(to_np(out)).astype(np.float64)
    valid = np.concatenate([np.arange(offsets[e], offsets[e] + counts[e]) for e in range(len(counts))])
    err = np.abs(got[valid] - h[valid])
    assert np.all(err <= bound[valid]), np.max(err / bound[valid])


def test_gemm_tiny_workload(gpu, O):
    """The tiny single-expert workload: x 64x256 with 1% x20 outliers (seed 0),
    W 128x256 ~N(0, 0.02^2); per-token x, per-expert W; out 64x128 fp32."""
    x = synth.normal_with_outliers(64, 256, seed=0, stream=0)
    w = synth.normal((1, 128, 256), seed=0, stream=1, std=0.02)
    xc, xs, xt = gpu.quantize_nvfp4_per_token(to_dev(x), swizzled=True)
    wc, ws, wt = gpu.quantize_nvfp4_per_expert(to_dev(w), swizzled=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu.grouped_expert_gemm_fp4(xc, xs, xt, to_dev(np.array([0, 64], np.int32)), wc, ws, wt,
                                      dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    oc, osf, ot = O.nvfp4_quantize_rows(x)
    wcc, wsf, wtt = O.nvfp4_quantize_group(w)
    ref, ab = O.gemm_nvfp4(oc, osf, ot, wcc[0], wsf[0], wtt[0])
    _assert_close(to_np(out), ref, ab)


def test_gemm_bad_offsets_reported(gpu, O):
    offsets, M, A, B = _make_problem(O, [128, 128], 256, 128, seed=4)
    bad = offsets.copy()
    bad[1] = 100  # a segment start that is not a multiple of 128
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ac, asf, at = A
    bc, bsf, bt = B
    gpu.grouped_expert_gemm_fp4(to_dev(ac), to_dev(O.sf_to_swizzled(asf)), to_dev(at), to_dev(bad), to_dev(bc),
                                to_dev(O.sf_to_swizzled(bsf.reshape(-1, bsf.shape[-1]))), to_dev(bt),
                                dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == gpu.DEV_BAD_OFFSETS


def test_gemm_many_experts_offsets_in_global(gpu, O):
    """More experts than the kernel caches in shared memory (its expert lookup
    then reads the offsets from global memory)."""
    counts = [(7 * e) % 40 for e in range(300)]
    offsets, M, A, B = _make_problem(O, counts, 128, 128, seed=21)
    out = _run(gpu, O, offsets, A, B, gpu.EPI_F32)
    ref, ab = _reference(O, offsets, A, B)
    _assert_close(to_np(out), ref, ab)


@pytest.mark.parametrize("epilogue", ["f32", "bf16"])
def test_gemm_capacity_not_tile_aligned(gpu, O, epilogue):
    """Segment starts are multiples of 128 but the capacity (and the last
    segment) ends mid-tile: rows past the capacity are neither read nor
    written."""
    counts, K, N = [100, 72], 320, 256
    offsets, M, A, B = _make_problem(O, counts, K, N, seed=31)
    cap = int(offsets[1]) + counts[1]                       # 200: ends inside the second tile
    ac, asf, at = A
    A2 = (ac[:cap], asf[:cap], at[:cap])
    offsets2 = offsets.copy()
    offsets2[-1] = cap
    # the SF buffer still holds whole 128-row tiles (swizzled layout)
    bc, bsf, bt = B
    E = bc.shape[0]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    epi = gpu.EPI_F32 if epilogue == "f32" else gpu.EPI_BF16
    out = gpu.grouped_expert_gemm_fp4(to_dev(A2[0]), to_dev(O.sf_to_swizzled(A2[1])), to_dev(A2[2]),
                                      to_dev(offsets2), to_dev(bc), to_dev(O.sf_to_swizzled(bsf.reshape(E * N, -1))),
                                      to_dev(bt), epilogue=epi, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert out.shape[0] == cap
    ref, ab = _reference(O, offsets2, A2, B)
    got = to_np(out) if epilogue == "f32" else synth.bf16_bits_to_f32(to_np(out))
    _assert_close(got, ref, ab, extra=0.0 if epilogue == "f32" else 2.0 ** -8)


# ---- many ragged experts: odd and even tile counts, empty experts, K tails
# (K % 256 != 0), segments of one row, and all three epilogues.

_RAGGED_CASES = [
    # counts, K, N: odd and even tile counts, empty experts, K tails (K % 256 != 0)
    ([300, 1, 0, 129, 385, 128, 256, 50], 320, 512),
    ([1000, 3, 700], 2048, 256),
    ([129] * 9, 576, 768),
]


@pytest.mark.parametrize("counts,K,N", _RAGGED_CASES)
@pytest.mark.parametrize("epilogue", ["f32", "bf16"])
def test_gemm_ragged_experts(gpu, O, counts, K, N, epilogue):
    offsets, M, A, B = _make_problem(O, counts, K, N, seed=sum(counts) + N)
    out = _run(gpu, O, offsets, A, B, gpu.EPI_F32 if epilogue == "f32" else gpu.EPI_BF16)
    ref, ab = _reference(O, offsets, A, B)
    got = to_np(out) if epilogue == "f32" else synth.bf16_bits_to_f32(to_np(out))
    _assert_close(got, ref, ab, extra=0.0 if epilogue == "f32" else 2.0 ** -8)


def test_gemm_swiglu_ragged_experts(gpu, O):
    counts, K, I = [300, 1, 0, 129, 385, 50], 320, 384
    offsets, M, A, B = _make_problem(O, counts, K, 2 * I, seed=77)
    out = _run(gpu, O, offsets, A, B, gpu.EPI_SWIGLU_BF16)
    ref, ab = _reference(O, offsets, A, B)
    h = O.swiglu(ref)
    g, u = ref[:, :I], ref[:, I:]
    dg, du = REL_ABS * ab[:, :I], REL_ABS * ab[:, I:]
    sg = g / (1 + np.exp(-g))
    bound = 1.1 * np.abs(u) * dg + np.abs(sg) * du + 2.0 ** -8 * np.abs(h) + 1e-30
    got = synth.bf16_bits_to_f32(to_np(out)).astype(np.float64)
    valid = np.concatenate([np.arange(offsets[e], offsets[e] + counts[e]) for e in range(len(counts))])
    err = np.abs(got[valid] - h[valid])
    assert np.all(err <= bound[valid]), np.max(err / bound[valid])


@pytest.mark.parametrize("epilogue", ["f32", "bf16"])
def test_gemm_capacity_ends_mid_tile_after_full_tiles(gpu, O, epilogue):
    """Three full tiles, then a last tile that ends at a capacity of 456 rows
    (mid-tile): rows past the capacity are neither read nor written."""
    counts, K, N = [300, 72], 320, 256
    offsets, M, A, B = _make_problem(O, counts, K, N, seed=41)
    cap = int(offsets[1]) + counts[1]
    ac, asf, at = A
    A2 = (ac[:cap], asf[:cap], at[:cap])
    offsets2 = offsets.copy()
    offsets2[-1] = cap
    bc, bsf, bt = B
    E = bc.shape[0]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    epi = gpu.EPI_F32 if epilogue == "f32" else gpu.EPI_BF16
    out = gpu.grouped_expert_gemm_fp4(to_dev(A2[0]), to_dev(O.sf_to_swizzled(A2[1])), to_dev(A2[2]),
                                      to_dev(offsets2), to_dev(bc), to_dev(O.sf_to_swizzled(bsf.reshape(E * N, -1))),
                                      to_dev(bt), epilogue=epi, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert out.shape[0] == cap
    ref, ab = _reference(O, offsets2, A2, B)
    got = to_np(out) if epilogue == "f32" else synth.bf16_bits_to_f32(to_np(out))
    _assert_close(got, ref, ab, extra=0.0 if epilogue == "f32" else 2.0 ** -8)


def test_gemm_bad_offsets_reported_wide_n(gpu, O):
    offsets, M, A, B = _make_problem(O, [256, 256], 256, 256, seed=5)
    bad = offsets.copy()
    bad[1] = 200
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ac, asf, at = A
    bc, bsf, bt = B
    gpu.grouped_expert_gemm_fp4(to_dev(ac), to_dev(O.sf_to_swizzled(asf)), to_dev(at), to_dev(bad), to_dev(bc),
                                to_dev(O.sf_to_swizzled(bsf.reshape(-1, bsf.shape[-1]))), to_dev(bt),
                                dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == gpu.DEV_BAD_OFFSETS
