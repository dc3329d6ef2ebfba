"""Oracle pins for the element and scale formats, the stochastic-rounding
rule and the Philox generator (CPU only)."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import golden

E2M1_VALUES = golden("page_examples.json")["nvfp4_value_set"]["magnitudes"]


def _brute_nearest(a, grid):
    """Nearest grid value by exhaustive comparison, ties to the even index."""
    best = None
    for i, g in enumerate(grid):
        d = abs(a - g)
        if best is None or d < best[0] or (d == best[0] and i % 2 == 0):
            best = (d, i)
    return best[1]


def test_e2m1_value_set_is_the_pages(O):
    mags = [O.e2m1_decode(c) for c in range(8)]
    assert mags == E2M1_VALUES
    assert [O.e2m1_decode(c | 8) for c in range(8)] == [-m for m in E2M1_VALUES]
    assert math.copysign(1.0, O.e2m1_decode(8)) == -1.0


def test_e2m1_roundtrip_all_codes(O):
    for c in range(16):
        assert O.e2m1_encode(O.e2m1_decode(c)) == c


def test_e2m1_encode_matches_brute_force(O):
    g = np.random.default_rng(11)
    vals = list(g.uniform(-8, 8, 20000).astype(np.float32))
    mids = [(a + b) / 2 for a, b in zip(E2M1_VALUES, E2M1_VALUES[1:])]
    for m in mids + E2M1_VALUES:
        for d in (0.0, 1e-6, -1e-6):
            vals += [np.float32(m + d), np.float32(-(m + d))]
    vals += [np.float32(x) for x in (6.0, 6.5, 7.0, 1e30, -1e30, 5.0, 3.5, 2.5, 0.25, 0.75)]
    codes = O.e2m1_encode_array(np.array(vals, np.float32))
    for v, c in zip(vals, codes):
        a = abs(float(v))
        idx = 7 if a >= 6.0 else _brute_nearest(a, E2M1_VALUES)
        sign = 8 if math.copysign(1.0, float(v)) < 0 else 0
        assert int(c) == (sign | idx), (v, c)


def test_e2m1_ties_go_to_even_code(O):
    # midpoints between neighbours: the even code wins
    expect = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for v, r in expect.items():
        assert O.e2m1_decode(O.e2m1_encode(v)) == r
        assert O.e2m1_decode(O.e2m1_encode(-v)) == -r


def test_e4m3_table_against_torch_float8(O):
    codes = torch.arange(256, dtype=torch.int16).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    for c in range(256):
        v = O.e4m3_decode(c)
        if c & 0x7F == 0x7F:
            assert math.isnan(v) and math.isnan(ref[c])
        else:
            assert v == ref[c] and math.copysign(1, v) == math.copysign(1, ref[c]), c
    assert O.e4m3_decode(0x7E) == 448.0
    assert O.e4m3_decode(0x01) == 2.0 ** -9
    assert O.e4m3_decode(0x08) == 2.0 ** -6


def test_e4m3_roundtrip_all_codes(O):
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert O.e4m3_encode(O.e4m3_decode(c)) == c


def test_e4m3_encode_against_torch_rne(O):
    g = np.random.default_rng(12)
    v = np.concatenate([
        g.uniform(-460, 460, 50000),
        np.exp2(g.uniform(-14, 9, 50000)) * g.choice([-1, 1], 50000),
    ]).astype(np.float32)
    # every midpoint between adjacent E4M3 values (ties must go to even)
    pos = np.array([O.e4m3_decode(c) for c in range(0x7F)], np.float64)
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids]).astype(np.float32)
    v = v[np.abs(v) < 448.0]
    ours = O.e4m3_encode_array(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturates_at_448(O):
    for v in (448.0, 449.0, 463.9, 464.0, 480.0, 1e6, 3.0e38):
        assert O.e4m3_encode(v) == 0x7E
        assert O.e4m3_encode(-v) == 0xFE


def test_e8m0_is_power_of_two(O):
    for c in range(255):
        assert O.e8m0_decode(c) == 2.0 ** (c - 127)
    assert math.isnan(O.e8m0_decode(255))


def test_philox_known_answers(O):
    kat = golden("philox4x32_10_kat.json")["vectors"]
    for v in kat:
        ctr = [int(x, 16) for x in v["ctr"]]
        key = [int(x, 16) for x in v["key"]]
        out = [int(x, 16) for x in v["out"]]
        assert list(O.philox4x32_10(ctr, key)) == out


def test_sr_bits_mapping_and_uniformity(O):
    # the 8 elements of one counter block read the 8 halves of one output
    seed = 0x0123456789ABCDEF
    words = O.philox4x32_10([5, 0, 1, 0], [seed & 0xFFFFFFFF, seed >> 32])
    halves = []
    for w in words:
        halves += [int(w) & 0xFFFF, int(w) >> 16]
    assert [O.sr_bits16(seed, 1, 40 + i) for i in range(8)] == halves
    # bit frequencies of a long stream are close to 1/2
    bits = np.array([O.sr_bits16(7, 0, i) for i in range(40000)], np.uint32)
    freq = [(bits >> b & 1).mean() for b in range(16)]
    assert all(abs(f - 0.5) < 0.02 for f in freq)


def test_sr_probability_is_distance_rule(O):
    # For grid-interior values, P(up) = ceil(f * 65536) / 65536, checked
    # exhaustively over all 65536 values of the random bits.
    cases = [(2.25, 2.0, 3.0), (0.3, 0.0, 0.5), (4.5, 4.0, 6.0), (1.1, 1.0, 1.5)]
    r = np.arange(65536, dtype=np.uint32)
    for v, lo, hi in cases:
        ups = sum(O.e2m1_decode(O.e2m1_encode_sr(v, int(x))) == hi for x in r[::97])
        f = Fraction(float(np.float32(v))) - Fraction(lo)
        f /= Fraction(hi - lo)
        p = math.ceil(f * 65536) / 65536
        n = len(r[::97])
        assert abs(ups / n - p) < 4 * math.sqrt(p * (1 - p) / n) + 2 / n
        assert O.e2m1_decode(O.e2m1_encode_sr(v, 0)) == (hi if f > 0 else lo)
        assert O.e2m1_decode(O.e2m1_encode_sr(v, 65535)) == lo
    # grid points never move
    for m in E2M1_VALUES:
        for x in (0, 1, 32767, 65535):
            assert O.e2m1_decode(O.e2m1_encode_sr(m, x)) == m
    # E4M3: between 1.0 and 1.125, 1.03125 is a quarter of the way
    assert O.e4m3_decode(O.e4m3_encode_sr(1.03125, 16383)) == 1.125
    assert O.e4m3_decode(O.e4m3_encode_sr(1.03125, 16384)) == 1.0
    assert O.e4m3_encode_sr(500.0, 0) == 0x7E


def test_sr_mean_preserving_e4m3(O):
    g = np.random.default_rng(3)
    vals = g.uniform(0.01, 400, 40)
    for v in vals:
        v = float(np.float32(v))
        draws = [O.e4m3_decode(O.e4m3_encode_sr(v, O.sr_bits16(9, 1, i))) for i in range(4000)]
        c = O.e4m3_encode(v)
        step = abs(O.e4m3_decode(c + 1) - O.e4m3_decode(c)) if c < 0x7E else 32
        assert abs(np.mean(draws) - v) < 0.05 * step


def test_bf16_rounding_from_f64(O):
    # exact rational checks of round-to-nearest-even into 8 significant bits
    cases = {
        1.0 + 2 ** -8: 1.0,                       # tie -> even
        1.0 + 3 * 2 ** -8: 1.0 + 2 ** -6,         # tie -> even (up)
        1.0 + 2 ** -8 + 2 ** -40: 1.0 + 2 ** -7,  # just above the tie
        -3.0 * 2 ** -9: -1.5 * 2 ** -8,           # exactly representable
    }
    for v, r in cases.items():
        b = O.f64_to_bf16(v)
        got = np.array([b], np.uint16).astype(np.uint32) << 16
        assert float(got.view(np.float32)[0]) == r
    assert O.f64_to_bf16(3.0e39) == 0x7F80
    assert O.f64_to_bf16(-0.0) == 0x8000
    # bf16 subnormal grid 2^-133
    assert O.f64_to_bf16(2.0 ** -133) == 0x0001
    assert O.f64_to_bf16(2.0 ** -134) == 0x0000     # tie -> even (0)
    assert O.f64_to_bf16(3 * 2.0 ** -134) == 0x0002  # tie -> even (2)
