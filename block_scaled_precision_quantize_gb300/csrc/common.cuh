// common.cuh -- device helpers shared by the block-scaled quantization kernels:
// bf16 bit handling, E2M1 / E4M3 / E8M0 conversions, the swizzled scale-factor
// layout, the Philox4x32-10 counter-based generator and device status words.
//
// Numerics: scale arithmetic uses the IEEE round-to-nearest intrinsics
// (__fdiv_rn, __frcp_rn, __fmul_rn, __fadd_rn, __fsub_rn) so that no FMA
// contraction or approximate division changes a bit; the library is built
// without fast math and without flush-to-zero.  This is the pages' rule that
// the FP4 quantizer must not use fast math ("LMSYS Drops Miles ...", section
// "The bit-exact quantizer contract").
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <stdint.h>

#include "../../include/bsq.h"

#define BSQ_DEVICE __device__ __forceinline__

namespace bsq {

constexpr float kNvfp4ScaleDivisor = 2688.0f;  // 6 (E2M1 max) * 448 (E4M3 max)
constexpr float kFltMax = 3.402823466e+38f;

// ---------------------------------------------------------------- status
// Programmatic dependent launch: wait until the grid this one depends on has
// completed (its writes visible), then let the next grid in the stream start
// its launch.  Both are no-ops when the kernel was launched without the
// programmatic-serialization attribute.
BSQ_DEVICE void pdl_enter()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

BSQ_DEVICE void report(int32_t* dev_status, int32_t code)
{
    if (dev_status != nullptr) atomicCAS(dev_status, BSQ_DEV_OK, code);
}

// ---------------------------------------------------------------- bf16
// bf16 bits -> binary32 (exact widening)
BSQ_DEVICE float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
BSQ_DEVICE float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// max |x| of the two bf16 values in a word, as a 16-bit magnitude pattern
// (for finite values the bit pattern orders like the magnitude)
BSQ_DEVICE uint32_t absmax_bf16x2(uint32_t acc, uint32_t w) { return __vmaxu2(acc, w & 0x7FFF7FFFu); }
BSQ_DEVICE uint32_t fold_halves(uint32_t m) { return max(m & 0xFFFFu, m >> 16); }
BSQ_DEVICE float bf16mag_to_f32(uint32_t m16) { return __uint_as_float(m16 << 16); }

// ---------------------------------------------------------------- host helpers
// Kernel attributes (the dynamic shared-memory opt-in) belong to each device's
// copy of the kernel: run `set` once per device of the calling thread, and
// again after a failure.  `done` is a bit per device id (ids >= 64 always run
// `set`).
template <class F>
inline cudaError_t once_per_device(std::atomic<uint64_t>& done, F set)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0u;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    err = set();
    if (err == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return err;
}

// ---------------------------------------------------------------- E2M1
// Eight binary32 values -> eight E2M1 codes packed in a word (element i in
// nibble i), round to nearest even, saturating at 6 (cvt ... satfinite).
BSQ_DEVICE uint32_t e2m1x8(float v0, float v1, float v2, float v3, float v4, float v5, float v6, float v7)
{
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
    return r;
}

// E2M1 code (low nibble) -> binary32, from the format definition:
// magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 is the sign.
BSQ_DEVICE float e2m1_to_f32(uint32_t nib)
{
    uint32_t em = nib & 7u;
    uint32_t bits = (em < 2u) ? (em ? 0x3F000000u : 0u) : ((((em >> 1) + 126u) << 23) | ((em & 1u) << 22));
    return __uint_as_float(bits | ((nib & 8u) << 28));
}

// Eight E2M1 codes (nibble i = element i) times one E4M3 scale factor, as
// four f16x2 pairs (element 2i in the low half of h[i]), exactly: E2M1 and
// E4M3 values are f16 values, and their product has at most 6 significant
// bits and magnitude in [2^-10, 2688], so the f16 multiply does not round.
BSQ_DEVICE void e2m1x8_scaled_f16x2(uint32_t w, uint32_t sf_byte, uint32_t (&h)[4])
{
    uint32_t s2;
    asm("{\n\t.reg .b16 b;\n\tcvt.u16.u32 b, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, b;\n\t}" : "=r"(s2) : "r"(sf_byte * 0x101u));
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
#pragma unroll
    for (int i = 0; i < 4; ++i) asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h[i]) : "r"(s2));
}
// d[j] = rn(rn(e2m1_j * sf) * t) for the eight codes of w (the inner product
// is exact, see above).
BSQ_DEVICE void e2m1x8_dequant(uint32_t w, uint32_t sf_byte, float t, float (&d)[8])
{
    uint32_t h[4];
    e2m1x8_scaled_f16x2(w, sf_byte, h);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
        d[2 * i] = __fmul_rn(f.x, t);
        d[2 * i + 1] = __fmul_rn(f.y, t);
    }
}

// ---------------------------------------------------------------- E4M3
// Four binary32 values -> four E4M3 bytes (element i in byte i), RNE satfinite.
BSQ_DEVICE uint32_t e4m3x4(float v0, float v1, float v2, float v3)
{
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
    return r;
}
BSQ_DEVICE uint32_t e4m3_rn(float v) { return e4m3x4(v, 0.f, 0.f, 0.f) & 0xFFu; }

// E4M3 byte -> binary32, from the format definition (bias 7, subnormals
// m * 2^-9).  The NaN codes are outside the contract.
BSQ_DEVICE float e4m3_to_f32(uint32_t c)
{
    uint32_t s = (c & 0x80u) << 24, e = (c >> 3) & 15u, m = c & 7u;
    float mag = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : __fmul_rn((float)m, 0.001953125f);
    return __uint_as_float(__float_as_uint(mag) | s);
}

// ---------------------------------------------------------------- SF layout
// Offset of scale factor (row, col) in the swizzled tile layout (tiles of 128
// rows x 4 columns, 512 bytes, tile-row major; inside a tile
// (r%32)*16 + (r/32)*4 + c%4).  ncol_tiles = ceil(SF columns / 4).
BSQ_DEVICE int64_t sf_swizzled(int64_t row, int64_t col, int64_t ncol_tiles)
{
    int64_t r = row & 127;
    return ((row >> 7) * ncol_tiles + (col >> 2)) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (col & 3);
}

// ---------------------------------------------------------------- Philox
// Philox4x32 with 10 rounds (Salmon et al., SC'11): per round the counter
// words 0 and 2 are multiplied by the two round constants (32x32 -> 64), the
// high halves are xored with the other words and the key; the key is bumped
// by the two Weyl constants between rounds.
BSQ_DEVICE uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t p0_lo = 0xD2511F53u * c.x, p0_hi = __umulhi(0xD2511F53u, c.x);
        const uint32_t p2_lo = 0xCD9E8D57u * c.z, p2_hi = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(p2_hi ^ c.y ^ k0, p2_lo, p0_hi ^ c.w ^ k1, p0_lo);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Philox4x32-10 with the round keys precomputed (k0 + r * 0x9E3779B9,
// k1 + r * 0xBB67AE85 for round r), passed by value as a kernel parameter:
// the same function as philox4x32_10, without the key schedule in the loop.
struct PhiloxKeys {
    uint32_t k0[10], k1[10];
};
inline PhiloxKeys philox_keys(uint64_t seed)
{
    PhiloxKeys k;
    uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
    for (int r = 0; r < 10; ++r, a += 0x9E3779B9u, b += 0xBB67AE85u) {
        k.k0[r] = a;
        k.k1[r] = b;
    }
    return k;
}
BSQ_DEVICE uint4 philox4x32_10_keys(uint4 c, const PhiloxKeys& k)
{
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c.x, p2 = (uint64_t)0xCD9E8D57u * c.z;
        c = make_uint4((uint32_t)(p2 >> 32) ^ c.y ^ k.k0[r], (uint32_t)p2, (uint32_t)(p0 >> 32) ^ c.w ^ k.k1[r],
                       (uint32_t)p0);
    }
    return c;
}
BSQ_DEVICE uint4 sr_block_bits_keys(const PhiloxKeys& k, uint32_t stream, uint64_t g)
{
    return philox4x32_10_keys(make_uint4((uint32_t)g, (uint32_t)(g >> 32), stream, 0u), k);
}

// Random bits for 8 consecutive elements 8g .. 8g+7 of a stream: element
// 8g + i takes the 16-bit half (i & 1) of word (i >> 1).
BSQ_DEVICE uint4 sr_block_bits(uint64_t seed, uint32_t stream, uint64_t g)
{
    return philox4x32_10(make_uint4((uint32_t)g, (uint32_t)(g >> 32), stream, 0u), (uint32_t)seed,
                         (uint32_t)(seed >> 32));
}
BSQ_DEVICE uint32_t sr_pick16(uint4 w, int i)
{
    uint32_t word = (i >> 1) == 0 ? w.x : (i >> 1) == 1 ? w.y : (i >> 1) == 2 ? w.z : w.w;
    return (i & 1) ? (word >> 16) : (word & 0xFFFFu);
}

// ---------------------------------------------------------------- SR encoders
// Stochastic rounding with 16 random bits r: with lo <= |v| < hi the two
// neighbouring grid points, round up iff r < 65536 * (|v| - lo) / (hi - lo);
// |v| >= max saturates.  Where the grid spacing is the binary32 spacing of
// |v| shifted by s bits (the normal ranges), (|v| - lo) / (hi - lo) * 65536
// equals (the s dropped bits) / 2^(s-16), so "round up" is a carry out of
// those bits after adding 2^s - 1 - (r << (s-16)).  Below the normal range the grid is uniform, g * 2^-s' (E2M1: 0.5 below 1;
// E4M3: 2^-9 below 2^-6), and X = |v| * 2^(s'+16) is exact.  With
// C = ceil(X) = 65536 k + c: rounding up iff r < f * 65536 (f the fraction of
// |v| / 2^-s') is, for an integer r, the carry out of c + 65535 - r, so the
// code is (C + 65535 - r) >> 16.  Both formulas can only overshoot the
// largest finite code from above, so saturation is a min.
BSQ_DEVICE uint32_t sr_uniform_code(float a, float scale_2p, uint32_t r16)
{
    uint32_t c;
    asm("cvt.rpi.u32.f32 %0, %1;" : "=r"(c) : "f"(__fmul_rn(a, scale_2p)));
    return (c + (0xFFFFu - r16)) >> 16;
}
BSQ_DEVICE uint32_t e2m1_sr(float v, uint32_t r16)
{
    const uint32_t bits = __float_as_uint(v), abits = bits & 0x7FFFFFFFu;
    // [1, 6): one mantissa bit kept (codes 2 .. 7 from the binary32 exponent and top bit)
    const uint32_t normal = ((abits + (0x3FFFFFu - (r16 << 6))) >> 22) - 252u;
    // [0, 1): grid 0.5 (codes 0, 1, 2), X = |v| * 2^17
    const uint32_t low = sr_uniform_code(__uint_as_float(abits), 131072.0f, r16);
    const uint32_t code = min(abits < 0x3F800000u ? low : normal, 7u);
    return ((bits >> 28) & 8u) | code;
}
BSQ_DEVICE uint32_t e4m3_sr(float v, uint32_t r16)
{
    const uint32_t bits = __float_as_uint(v), abits = bits & 0x7FFFFFFFu;
    // normal range [2^-6, 448): three mantissa bits kept; code = ((e - 120) << 3) | m
    const uint32_t normal = ((abits + (0xFFFFFu - (r16 << 4))) >> 20) - 960u;
    // [0, 2^-6): grid 2^-9 (codes 0 .. 8), X = |v| * 2^25
    const uint32_t low = sr_uniform_code(__uint_as_float(abits), 33554432.0f, r16);
    const uint32_t code = min(abits < 0x3C800000u ? low : normal, 0x7Eu);
    return ((bits >> 24) & 0x80u) | code;
}

// ---------------------------------------------------------------- NVFP4 block
// Scale math of one 16-element block (see quantize_nvfp4_per_token):
// s = E4M3(rn(amax_b / rn(mult * t))), d = rn(decode(s) * t),
// enc = d == 0 ? 0 : rn(1 / d) (infinite -> FLT_MAX).
struct BlockScale {
    uint32_t sf;
    float d;
    float enc;
};
BSQ_DEVICE BlockScale nvfp4_block_scale(float amax_b, float mult_t, float t)
{
    BlockScale b;
    b.sf = e4m3_rn(__fdiv_rn(amax_b, mult_t));
    b.d = __fmul_rn(e4m3_to_f32(b.sf), t);
    float enc = (b.d == 0.0f) ? 0.0f : __frcp_rn(b.d);
    b.enc = isinf(enc) ? kFltMax : enc;
    return b;
}

// Eight E2M1 codes (nibble i = element i) decoded to binary32 with the
// hardware conversion to f16 pairs (exact: E2M1 values are f16 values).
BSQ_DEVICE void e2m1x8_to_f32(uint32_t w, float* v)
{
    uint32_t h[4];
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
// Squared error of a candidate block (codes packed 8 per word), summed by the
// fixed tree p_j = s_j + s_{j+8}, q_j = p_j + p_{j+4}, r_j = q_j + q_{j+2}.
BSQ_DEVICE float block_sse(const float x[16], uint32_t c_lo, uint32_t c_hi, float d)
{
    float v[16], sq[16];
    e2m1x8_to_f32(c_lo, v);
    e2m1x8_to_f32(c_hi, v + 8);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float e = __fsub_rn(x[i], __fmul_rn(v[i], d));
        sq[i] = __fmul_rn(e, e);
    }
    float p[8], q[4];
#pragma unroll
    for (int j = 0; j < 8; ++j) p[j] = __fadd_rn(sq[j], sq[j + 8]);
#pragma unroll
    for (int j = 0; j < 4; ++j) q[j] = __fadd_rn(p[j], p[j + 4]);
    return __fadd_rn(__fadd_rn(q[0], q[2]), __fadd_rn(q[1], q[3]));
}
BSQ_DEVICE uint2 encode16(const float x[16], float enc)
{
    float q[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = __fmul_rn(x[i], enc);
    return make_uint2(e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]),
                      e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]));
}

// MXFP8 shared exponent from the bit pattern of a block maximum (> 0):
// X = clamp(floor(log2 amax) - 8, -127, 127); returns X.
// ---------------------------------------------------------------- NVFP4 block
// max |x| of 16 bf16 values (two 16-byte words) as a bf16 magnitude pattern
BSQ_DEVICE uint32_t absmax16(const uint4& a, const uint4& b)
{
    uint32_t m = absmax_bf16x2(0u, a.x);
    m = absmax_bf16x2(m, a.y);
    m = absmax_bf16x2(m, a.z);
    m = absmax_bf16x2(m, a.w);
    m = absmax_bf16x2(m, b.x);
    m = absmax_bf16x2(m, b.y);
    m = absmax_bf16x2(m, b.z);
    m = absmax_bf16x2(m, b.w);
    return fold_halves(m);
}

BSQ_DEVICE void unpack16(const uint4& a, const uint4& b, float x[16])
{
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        x[2 * i] = bf16_lo(w[i]);
        x[2 * i + 1] = bf16_hi(w[i]);
    }
}

// One 16-element block of bf16 -> E2M1 codes (2 words) and the E4M3 block
// scale byte, given the row (or tensor) scale t: the per-token recipe, with
// the 4/6 choice of block scale when FOUR_SIX.  Shared by the quantizers and
// the grouped GEMM's fused quantization of h.
template <bool FOUR_SIX>
BSQ_DEVICE void nvfp4_block(const uint4& a, const uint4& b, uint32_t amax16_bits, float t, float six_t,
                            float four_t, uint2& codes, uint32_t& sf)
{
    if (t == 0.0f) {
        codes = make_uint2(0u, 0u);
        sf = 0u;
        return;
    }
    float x[16];
    unpack16(a, b, x);
    const float ab = bf16mag_to_f32(amax16_bits);
    const BlockScale s6 = nvfp4_block_scale(ab, six_t, t);
    codes = encode16(x, s6.enc);
    sf = s6.sf;
    if (FOUR_SIX) {
        const BlockScale s4 = nvfp4_block_scale(ab, four_t, t);
        const uint2 c4 = encode16(x, s4.enc);
        const float e6 = block_sse(x, codes.x, codes.y, s6.d);
        const float e4 = block_sse(x, c4.x, c4.y, s4.d);
        if (e4 < e6) {
            codes = c4;
            sf = s4.sf;
        }
    }
}

BSQ_DEVICE int mx_exponent(uint32_t amax_bits)
{
    const int e = (int)(amax_bits >> 23);
    return e == 0 ? -127 : max(e - 127 - 8, -127);
}
BSQ_DEVICE float mx_multiplier(int X) { return __uint_as_float((uint32_t)(127 - X) << 23); }  // 2^-X

}  // namespace bsq
