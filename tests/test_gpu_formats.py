"""GPU: the kernels' element conversions and random bits against the oracle
(bit-exact), over all codes and over dense sweeps of binary32 inputs."""
import numpy as np
import pytest
import torch

from conftest import bits_equal, first_mismatch, to_dev, to_np

pytestmark = pytest.mark.gpu


def _sweep_e2m1():
    """Every binary32 in [2^-4, 8) (all mantissas of 7 binades), both signs,
    plus zeros, subnormals, large values."""
    exps = np.arange(123, 130, dtype=np.uint32)  # 2^-4 .. 2^2 (values < 8)
    mant = np.arange(0, 1 << 23, 1, dtype=np.uint32)
    bits = (exps[:, None] << 23 | mant[None, :]).ravel()
    extra = np.array([0, 1, 2, 0x007FFFFF, 0x00800000, 0x3D000000, 0x40C00000, 0x40E00000, 0x41000000,
                      0x7F7FFFFF, 0x3E7FFFFF, 0x3E800000, 0x3E800001], np.uint32)
    bits = np.concatenate([bits, extra])
    bits = np.concatenate([bits, bits | np.uint32(0x80000000)])
    return bits.view(np.float32)


def test_e2m1_rne_exhaustive_sweep(gpu, O):
    v = _sweep_e2m1()
    got = to_np(gpu.format_probe(0, to_dev(v)))
    ref = O.e2m1_encode_array(v)
    assert bits_equal(got, ref), first_mismatch(got, ref)


def test_e4m3_rne_sweep(gpu, O):
    # all binary32 with exponent in [2^-11, 2^9) at mantissa stride 3, both signs
    exps = np.arange(116, 136, dtype=np.uint32)
    mant = np.arange(0, 1 << 23, 3, dtype=np.uint32)
    bits = (exps[:, None] << 23 | mant[None, :]).ravel()
    pos = np.array([O.e4m3_decode(c) for c in range(0x7F)], np.float64)
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32).view(np.uint32)
    extra = np.concatenate([mids, mids + 1, mids - 1, np.array([0, 1, 0x7F7FFFFF, 0x43E00000, 0x43E80000], np.uint32)])
    bits = np.concatenate([bits, extra])
    bits = np.concatenate([bits, bits | np.uint32(0x80000000)])
    v = bits.view(np.float32)
    got = to_np(gpu.format_probe(1, to_dev(v)))
    ref = O.e4m3_encode_array(v)
    assert bits_equal(got, ref), first_mismatch(got, ref)


def test_decodes_all_codes(gpu, O):
    c = np.arange(256, dtype=np.uint32)
    codes_as_f32 = c.view(np.float32)
    e2 = to_np(gpu.format_probe(4, to_dev(codes_as_f32[:16].copy())))
    assert bits_equal(e2, np.array([O.e2m1_decode(i) for i in range(16)], np.float32))
    keep = np.array([i for i in range(256) if i & 0x7F != 0x7F])
    e4 = to_np(gpu.format_probe(5, to_dev(codes_as_f32.copy())))
    assert bits_equal(e4[keep], np.array([O.e4m3_decode(i) for i in keep], np.float32))


@pytest.mark.parametrize("kind", [2, 3])
def test_stochastic_encoders(gpu, O, kind):
    g = np.random.default_rng(kind)
    n = 200000
    hi = 7.0 if kind == 2 else 470.0
    v = np.concatenate([g.uniform(-hi, hi, n),
                        np.exp2(g.uniform(-12, 9, n)) * g.choice([-1, 1], n)]).astype(np.float32)
    if kind == 2:
        grid = np.array([0, .25, .5, .75, 1, 1.25, 1.5, 1.75, 2, 2.5, 3, 3.5, 4, 5, 6], np.float32)
        v = np.concatenate([v, grid, -grid]).astype(np.float32)
    r = g.integers(0, 1 << 16, v.size).astype(np.uint32)
    r[:64] = 0
    r[64:128] = 0xFFFF
    got = to_np(gpu.format_probe(kind, to_dev(v), to_dev(r)))
    enc = O.e2m1_encode_sr if kind == 2 else O.e4m3_encode_sr
    idx = np.concatenate([np.arange(0, v.size, 7), np.arange(v.size - 40, v.size)])
    ref = np.array([enc(float(v[i]), int(r[i])) for i in idx], np.uint8)
    assert bits_equal(got[idx], ref), first_mismatch(got[idx], ref)


def _sr_boundary_cases(grid):
    """Values lo + (j / 65536) * (hi - lo) inside every grid interval, j at the
    carry boundaries, each with random bits j - 1, j and j + 1: rounding up is
    decided exactly at r = j."""
    vals, bits = [], []
    for lo, hi in zip(grid[:-1], grid[1:]):
        for j in (1, 2, 255, 256, 32767, 32768, 65535):
            v = np.float32(lo + (hi - lo) * (j / 65536.0))
            assert float(v) == lo + (hi - lo) * (j / 65536.0)      # exact in binary32
            for r in (j - 1, j, j + 1):
                if 0 <= r < 65536:
                    vals += [v, -v]
                    bits += [r, r]
    return np.array(vals, np.float32), np.array(bits, np.uint32)


@pytest.mark.parametrize("kind", [2, 3])
def test_stochastic_encoders_carry_boundaries(gpu, O, kind):
    if kind == 2:
        grid = [0, .5, 1, 1.5, 2, 3, 4, 6]
    else:
        grid = sorted({O.e4m3_decode(c) for c in range(0x7F)})   # 0 .. 448, subnormals included
    v, r = _sr_boundary_cases([float(g) for g in grid])
    got = to_np(gpu.format_probe(kind, to_dev(v), to_dev(r)))
    enc = O.e2m1_encode_sr if kind == 2 else O.e4m3_encode_sr
    ref = np.array([enc(float(a), int(b)) for a, b in zip(v, r)], np.uint8)
    assert bits_equal(got, ref), first_mismatch(got, ref)


def test_philox_bits_match_oracle(gpu, O):
    for seed, stream, idx0 in [(7, 0, 0), (7, 1, 0), (0xDEADBEEFCAFEF00D, 1, (1 << 35) - 13), (123, 0, 999)]:
        n = 4096
        got = to_np(gpu.philox_bits16(seed, stream, idx0, n))
        ref = np.array([O.sr_bits16(seed, stream, idx0 + i) for i in range(n)], np.uint16)
        assert bits_equal(got, ref), (seed, stream, idx0, first_mismatch(got, ref))
