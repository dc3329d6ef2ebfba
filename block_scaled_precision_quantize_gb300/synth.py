"""Seeded synthetic inputs for the block-scaled MoE workloads.

This module only draws random tensors with the shapes and value
distributions of the workloads (activations with outliers, rows of widely
varying scale, expert weights, top-k routing); it holds none of the
quantization or GEMM arithmetic, so both the CUDA path and the CPU oracle can
be fed from it without sharing any of the method.

bf16 tensors are produced by rounding binary32 normals to nearest even and
are returned as raw uint16 bit patterns (numpy) unless stated otherwise.

Workloads (sizes as the MoE pages quote them):
  tiny      x 64x256 ~N(0,1) with 1% of entries x20 (seed 0, stream 0),
            W 128x256 ~N(0, 0.02^2) (seed 0, stream 1)
  mxfp8     16384x2048, row r ~N(0, s_r^2), s_r = 10^U(-3, 2) (seed 2)
  qwen3     Qwen3-30B-A3B-shaped expert layer: T=16384, H=2048, E=128,
            top-8, I=768; x ~N(0,1) (seed 3), router logits ~N(0,1)
  requant   bf16 ~N(0,1) with 1% x20 outliers (seed 7), 16384x2048 and
            16384x768, to be NVFP4-quantized and then requantized
  deepseek  DeepSeek-V3-shaped expert layer: T=32768, H=7168, E=256, top-8,
            I=2048; router logits N(0,1) plus a Zipf(s=1.1) expert bias
  nvfp4     random NVFP4 operands (codes, block scales, FP32 scales) for the
            dequantization tests: uniform code bytes, block-scale bytes
            uniform over the non-negative finite E4M3 codes, log-normal scales
"""
from __future__ import annotations

import numpy as np

try:  # torch is only needed for bf16 rounding and device-side weights
    import torch
except ImportError:  # pragma: no cover
    torch = None


def rng(seed: int, stream: int = 0) -> np.random.Generator:
    """Independent numpy generator for (seed, stream)."""
    return np.random.default_rng([int(seed), int(stream)])


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round binary32 values to bf16 (nearest even); return uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to binary32."""
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_with_outliers(rows: int, cols: int, seed: int, stream: int = 0,
                         p_outlier: float = 0.01, factor: float = 20.0) -> np.ndarray:
    """bf16 bits of N(0,1) with each entry multiplied by `factor` w.p. p."""
    g = rng(seed, stream)
    x = g.standard_normal((rows, cols), dtype=np.float32)
    mask = g.random((rows, cols)) < p_outlier
    x[mask] *= np.float32(factor)
    return to_bf16_bits(x)


def normal(shape, seed: int, stream: int = 0, std: float = 1.0) -> np.ndarray:
    g = rng(seed, stream)
    x = g.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return to_bf16_bits(x)


def rows_log_uniform_std(rows: int, cols: int, seed: int, lo_exp: float = -3.0,
                         hi_exp: float = 2.0) -> np.ndarray:
    """bf16 bits; row r ~ N(0, s_r^2) with s_r = 10^U(lo_exp, hi_exp)."""
    g = rng(seed, 0)
    s = np.power(10.0, g.uniform(lo_exp, hi_exp, size=(rows, 1))).astype(np.float32)
    x = g.standard_normal((rows, cols), dtype=np.float32) * s
    return to_bf16_bits(x)


def special_rows(cols: int) -> np.ndarray:
    """Boundary rows for bit-exact tests: all zero, negative zeros, the bf16
    maximum, bf16 subnormals, exact E2M1 grid points and their midpoints, a
    single non-zero, alternating signs, huge dynamic range."""
    f = np.float32
    bmax = np.uint16(0x7F7F)
    rows = []
    rows.append(np.zeros(cols, np.uint16))
    rows.append(np.full(cols, 0x8000, np.uint16))
    rows.append(np.full(cols, bmax, np.uint16))
    r = np.full(cols, bmax, np.uint16)
    r[1::2] |= 0x8000
    rows.append(r)
    rows.append(np.arange(cols, dtype=np.uint16) % 0x7F + 1)  # bf16 subnormals
    grid = np.array([0, .25, .5, .75, 1, 1.25, 1.5, 1.75, 2, 2.5, 3, 3.5, 4, 5, 6, 7], f)
    rows.append(to_bf16_bits(np.resize(grid, cols)))
    rows.append(to_bf16_bits(-np.resize(grid, cols) * f(64)))
    one = np.zeros(cols, f)
    one[cols // 3] = f(-3.0e-3)
    rows.append(to_bf16_bits(one))
    wide = np.power(f(2.0), (np.arange(cols) % 60 - 30).astype(f)) * np.where(np.arange(cols) % 3 == 0, f(-1), f(1))
    rows.append(to_bf16_bits(wide))
    return np.stack(rows)


def topk_routing(T: int, E: int, k: int, seed: int, zipf_s: float | None = None):
    """Top-k routing from softmax of N(0,1) logits (plus an optional Zipf
    expert bias log p_e, p_e proportional to rank_e^-s over a seeded random
    ranking of the experts). Ties go to the lower expert id. Weights are the
    top-k probabilities renormalized to sum to 1.
    Returns (ids int32 [T, k], weights float32 [T, k])."""
    g = rng(seed, 0)
    logits = g.standard_normal((T, E), dtype=np.float32).astype(np.float64)
    if zipf_s is not None:
        ranks = g.permutation(E) + 1
        p = ranks.astype(np.float64) ** (-zipf_s)
        p /= p.sum()
        logits = logits + np.log(p)[None, :]
    z = logits - logits.max(axis=1, keepdims=True)
    prob = np.exp(z)
    prob /= prob.sum(axis=1, keepdims=True)
    order = np.argsort(-prob, axis=1, kind="stable")[:, :k]
    ids = order.astype(np.int32)
    w = np.take_along_axis(prob, order, axis=1)
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w


def device_normal_bf16(shape, seed: int, std: float, device="cuda"):
    """Large weight tensors drawn directly on the device (torch Philox
    generator seeded with `seed`), returned as a bf16 torch tensor."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    w = torch.empty(shape, dtype=torch.bfloat16, device=device)
    # draw in chunks of rows to bound the fp32 temporary
    flat = w.view(-1, shape[-1])
    step = max(1, (1 << 26) // shape[-1])
    for r0 in range(0, flat.shape[0], step):
        r1 = min(flat.shape[0], r0 + step)
        tmp = torch.randn((r1 - r0, shape[-1]), generator=gen, device=device, dtype=torch.float32)
        flat[r0:r1] = (tmp * std).to(torch.bfloat16)
    return w


WORKLOADS = {
    "tiny": dict(M=64, K=256, N=128, seed=0),
    "mxfp8": dict(rows=16384, K=2048, seed=2),
    "qwen3": dict(T=16384, H=2048, E=128, k=8, I=768, seed=3, w_std=0.02),
    "requant": dict(shapes=[(16384, 2048), (16384, 768)], seed=7),
    "deepseek": dict(T=32768, H=7168, E=256, k=8, I=2048, seed=5, w_std=0.02, zipf_s=1.1),
}


def random_nvfp4(rows: int, K: int, seed: int, groups: int | None = None):
    """Random NVFP4 operands: codes u8 [rows, K/2] (uniform bytes), block-scale
    bytes u8 [rows, K/16] uniform over 0x00..0x7E (the non-negative finite
    E4M3 codes, as the quantizers emit), and positive f32 scales, one per row
    (or per group when `groups` is given), log-normal around 2^-8."""
    g = rng(seed, 0)
    codes = g.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
    sf = g.integers(0, 0x7F, size=(rows, K // 16), dtype=np.uint8)
    n = rows if groups is None else groups
    scale = np.exp2(g.normal(-8.0, 3.0, size=n)).astype(np.float32)
    return codes, sf, scale

