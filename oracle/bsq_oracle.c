/*
 * bsq_oracle.c -- the oracle: a plain, slow, single-threaded CPU restatement
 * of what the block-scaled quantization hot path computes.
 *
 * TEST INFRASTRUCTURE ONLY. It is built and loaded by the tests, by the smoke
 * check and by the benchmark's CPU-baseline leg; the product library never
 * includes, links or calls it, and it includes nothing from the product.
 *
 * Sources (web pages; each function names the one it follows):
 *  [MILES-IT]  "Miles Blackwell RL sostituisce l'uniformita BF16 con MXFP8 e
 *              NVFP4 nativi" (remio.ai)
 *  [HUMANS-JP] "4ビットの教訓：NVFP4 RLにおける安定性とパフォーマンスのバランス"
 *              (hackernews.jp), section "ベースラインレシピ"
 *  [LMSYS]     "LMSYS Drops Miles, an Open-Source RL Framework Running 4x
 *              Faster on Blackwell GPUs" (alphasignal.ai)
 *  [TML-ZH]    "End-to-End 4-Bit Training" summary (nopree.com)
 *  [PHILOX]    Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
 *              as 1, 2, 3", SC'11 (the Philox-4x32 counter-based generator)
 *
 * Where the pages leave a step open, the reading taken is marked READING and
 * is the same reading the CUDA path implements.
 *
 * Floating point: every float expression below is a single binary32
 * operation rounded to nearest even (compiled with -ffp-contract=off, no fast
 * math, no flush-to-zero); fp64 is used only where stated.
 */
#include "bsq_oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define EXPORT __attribute__((visibility("default")))

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
/* bf16 is the upper half of a binary32; widening is exact. */
static float bf16_to_f32(uint16_t b) { return bits_to_f32((uint32_t)b << 16); }

/* ------------------------------------------------------------------------
 * E2M1 (the NVFP4 element).  [TML-ZH] section "先说为什么难": the only
 * magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6.  Code = sign bit (bit 3) and
 * the index of the magnitude in that list (bits 2..0).
 * Encoding is round-to-nearest with ties to the even code, saturating at 6.
 * READING: the sign of zero is kept (a negative input that rounds to zero
 * gives code 0x8), as IEEE conversions do.
 * ---------------------------------------------------------------------- */
static const float E2M1_MAG[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

EXPORT float bsqo_e2m1_decode(uint32_t code)
{
    float m = E2M1_MAG[code & 7u];
    return (code & 8u) ? -m : m;
}

EXPORT uint32_t bsqo_e2m1_encode(float v)
{
    uint32_t sign = signbit(v) ? 8u : 0u;
    float a = fabsf(v);
    uint32_t c = 0;
    if (a >= 6.0f) return sign | 7u;
    while (c < 7u && E2M1_MAG[c + 1] <= a) c++;         /* largest magnitude <= a */
    if (c < 7u) {
        float mid = 0.5f * (E2M1_MAG[c] + E2M1_MAG[c + 1]);   /* exact */
        if (a > mid || (a == mid && (c & 1u))) c++;          /* ties to even code */
    }
    return sign | c;
}

/* ------------------------------------------------------------------------
 * E4M3 (the NVFP4 block scale and the MXFP8 element): 1 sign, 4 exponent
 * bits (bias 7), 3 mantissa bits, no infinities, S.1111.111 is NaN, largest
 * finite 448, smallest subnormal 2^-9.  [MILES-IT] "Il supporto Miles ...":
 * NVFP4 keeps one E4M3 scale per 16 values; MXFP8 elements are E4M3.
 * The value of every code is computed from that definition; positive codes
 * 0x00..0x7E are increasing in value, so encoding is a search in that table.
 * ---------------------------------------------------------------------- */
static float e4m3_table[256];
static int e4m3_ready = 0;

static void e4m3_init(void)
{
    if (e4m3_ready) return;
    for (uint32_t c = 0; c < 256u; ++c) {
        uint32_t s = (c >> 7) & 1u, e = (c >> 3) & 15u, m = c & 7u;
        float mag;
        if (e == 15u && m == 7u) mag = NAN;
        else if (e == 0u) mag = ldexpf((float)m, -9);             /* subnormal: m * 2^-9 */
        else mag = ldexpf(1.0f + (float)m / 8.0f, (int)e - 7);  /* (1 + m/8) * 2^(e-7) */
        e4m3_table[c] = s ? -mag : mag;
    }
    e4m3_ready = 1;
}

EXPORT float bsqo_e4m3_decode(uint32_t code)
{
    e4m3_init();
    return e4m3_table[code & 0xFFu];
}

/* Largest positive code whose value is <= a (0 <= a < 448). */
static uint32_t e4m3_floor_code(float a)
{
    uint32_t lo = 0, hi = 0x7Eu;
    while (lo < hi) {                           /* binary search in the table */
        uint32_t mid = (lo + hi + 1u) / 2u;
        if (e4m3_table[mid] <= a) lo = mid; else hi = mid - 1u;
    }
    return lo;
}

/* Round to nearest, ties to even code; anything at or above 448 saturates to
 * 448 (the "satfinite" rule; config 2 of the workloads states "RNE
 * saturating at 448"). */
EXPORT uint32_t bsqo_e4m3_encode(float v)
{
    e4m3_init();
    uint32_t sign = signbit(v) ? 0x80u : 0u;
    float a = fabsf(v);
    if (a >= 448.0f) return sign | 0x7Eu;
    uint32_t c = e4m3_floor_code(a);
    float lo = e4m3_table[c], hi = e4m3_table[c + 1];
    float mid = 0.5f * (lo + hi);  /* exact: both share a power-of-two grid */
    if (a > mid || (a == mid && (c & 1u))) c++;
    return sign | c;
}

/* E8M0 (the MXFP8 block scale): value 2^(c-127); 0xFF is NaN.
 * [LMSYS] "Recipe 1: End-to-end MXFP8": 32 E4M3 values share one E8M0 scale. */
EXPORT float bsqo_e8m0_decode(uint32_t code)
{
    code &= 0xFFu;
    if (code == 0xFFu) return NAN;
    return ldexpf(1.0f, (int)code - 127);
}

EXPORT void bsqo_e2m1_encode_array(const float* v, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)bsqo_e2m1_encode(v[i]);
}

EXPORT void bsqo_e4m3_encode_array(const float* v, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)bsqo_e4m3_encode(v[i]);
}

/* ------------------------------------------------------------------------
 * Stochastic rounding.  [TML-ZH] section "第二个决定": instead of the nearest
 * value, round to one of the two neighbours with probability given by the
 * distance, so the expectation is unchanged.
 * READING (16 random bits per element): with lo <= |v| < hi the neighbouring
 * grid points and f = (|v| - lo) / (hi - lo) (exact in binary32: the grid
 * spacing is a power of two inside a binade), round up iff r16 < f * 65536,
 * r16 uniform in [0, 65536).  |v| at or above the largest value saturates.
 * ---------------------------------------------------------------------- */
EXPORT uint32_t bsqo_e2m1_encode_sr(float v, uint32_t r16)
{
    uint32_t sign = signbit(v) ? 8u : 0u;
    float a = fabsf(v);
    if (a >= 6.0f) return sign | 7u;
    uint32_t c = 0;
    while (c < 7u && E2M1_MAG[c + 1] <= a) c++;
    float lo = E2M1_MAG[c], hi = E2M1_MAG[c + 1];
    float f = (a - lo) / (hi - lo);
    if ((float)(r16 & 0xFFFFu) < f * 65536.0f) c++;
    return sign | c;
}

EXPORT uint32_t bsqo_e4m3_encode_sr(float v, uint32_t r16)
{
    e4m3_init();
    uint32_t sign = signbit(v) ? 0x80u : 0u;
    float a = fabsf(v);
    if (a >= 448.0f) return sign | 0x7Eu;
    uint32_t c = e4m3_floor_code(a);
    float lo = e4m3_table[c], hi = e4m3_table[c + 1];
    float f = (a - lo) / (hi - lo);
    if ((float)(r16 & 0xFFFFu) < f * 65536.0f) c++;
    return sign | c;
}

/* ------------------------------------------------------------------------
 * Philox-4x32 with 10 rounds [PHILOX].  State: four 32-bit counter words and
 * a two-word key.  One round multiplies counter words 0 and 2 by the two
 * round multipliers (0xD2511F53, 0xCD9E8D57) as 32x32->64 products; the new
 * words are (hi(word2 product) ^ word1 ^ key0, lo(word2 product),
 * hi(word0 product) ^ word3 ^ key1, lo(word0 product)).  Between rounds the
 * key is bumped by the Weyl constants (0x9E3779B9, 0xBB67AE85).
 * ---------------------------------------------------------------------- */
EXPORT void bsqo_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)x0;
        uint64_t p2 = (uint64_t)0xCD9E8D57u * (uint64_t)x2;
        uint32_t y0 = (uint32_t)(p2 >> 32) ^ x1 ^ k0;
        uint32_t y1 = (uint32_t)p2;
        uint32_t y2 = (uint32_t)(p0 >> 32) ^ x3 ^ k1;
        uint32_t y3 = (uint32_t)p0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* READING (how elements draw their bits): key = (low, high) 32-bit halves of
 * the seed; counter = (low, high) halves of g = idx / 8, then the stream id,
 * then 0.  Element idx takes 16-bit half (idx & 1) (0 = low half) of output
 * word ((idx >> 1) & 3).  idx is the linear index of the element in the
 * output tensor; stream 0 feeds the NVFP4 target and stream 1 the MXFP8 one. */
EXPORT uint32_t bsqo_sr_bits16(uint64_t seed, uint32_t stream, uint64_t idx)
{
    uint64_t g = idx >> 3;
    uint32_t ctr[4] = {(uint32_t)g, (uint32_t)(g >> 32), stream, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    bsqo_philox4x32_10(ctr, key, out);
    uint32_t w = out[(idx >> 1) & 3u];
    return (idx & 1u) ? (w >> 16) : (w & 0xFFFFu);
}

/* ------------------------------------------------------------------------
 * NVFP4 two-level quantization of one row.
 * [MILES-IT] "Il supporto Miles ...": E2M1 values, one E4M3 scale per block
 * of 16 values, plus a wider FP32 scale; Miles computes that FP32 scale per
 * token.  [HUMANS-JP] "ベースラインレシピ" and [LMSYS] "Recipe 2": each token
 * computes its own FP32 activation scale over the hidden dimension, online,
 * from the observed values, fused into the quantization kernel; weights keep
 * one FP32 scale per tensor ([TML-ZH] "工程细节": one outer scale per
 * expert).
 *
 * Steps (x already widened to binary32):
 *  1. amax = max |x|                         (exact)
 *  2. t = rn(amax / 2688)   READING: 2688 = 6 * 448 puts the largest block
 *     scale at the E4M3 maximum.  If t == 0 every code and SF byte is 0.
 *  3. per 16-block b, with candidate multiplier m (6; or 4 under "4/6"):
 *       s = E4M3(rn(amax_b / rn(m * t))),  d = rn(decode(s) * t)
 *  4. READING: elements use a reciprocal, enc = d == 0 ? 0 : rn(1 / d)
 *     (an infinite reciprocal becomes FLT_MAX); code = E2M1(rn(x * enc)).
 *  5. dequantization is rn(rn(value(code) * decode(s)) * t).
 * "4/6" ([TML-ZH] "工程细节": per block, pick one of two candidate scales to
 * reduce error; activations only).  READING: candidates m = 6 and m = 4;
 * block error e_i = rn(x_i - rn(value(code_i) * d)), sq_i = rn(e_i * e_i),
 * summed by the fixed tree p_j = sq_j + sq_{j+8}, q_j = p_j + p_{j+4},
 * r_j = q_j + q_{j+2}, S = r_0 + r_1; m = 4 wins only if S4 < S6.
 * ---------------------------------------------------------------------- */
static void nvfp4_block_candidate(const float* x, float t, float mult,
                                  uint8_t* code16, uint8_t* sf_out, float* sse_out)
{
    float amax_b = 0.0f;
    for (int i = 0; i < 16; ++i) amax_b = fmaxf(amax_b, fabsf(x[i]));
    float denom = mult * t;
    float s_raw = amax_b / denom;
    uint32_t s = bsqo_e4m3_encode(s_raw);
    float d = bsqo_e4m3_decode(s) * t;
    float enc = (d == 0.0f) ? 0.0f : 1.0f / d;
    if (isinf(enc)) enc = FLT_MAX;
    float sq[16];
    for (int i = 0; i < 16; ++i) {
        float q = x[i] * enc;
        code16[i] = (uint8_t)bsqo_e2m1_encode(q);
        float rec = bsqo_e2m1_decode(code16[i]) * d;
        float e = x[i] - rec;
        sq[i] = e * e;
    }
    float p[8], qq[4], r[2];
    for (int j = 0; j < 8; ++j) p[j] = sq[j] + sq[j + 8];
    for (int j = 0; j < 4; ++j) qq[j] = p[j] + p[j + 4];
    for (int j = 0; j < 2; ++j) r[j] = qq[j] + qq[j + 2];
    *sse_out = r[0] + r[1];
    *sf_out = (uint8_t)s;
}

static void nvfp4_row_given_t(const float* x, int64_t K, float t, int four_six,
                              uint8_t* codes, uint8_t* sf)
{
    if (t == 0.0f) {
        memset(codes, 0, (size_t)(K / 2));
        memset(sf, 0, (size_t)(K / 16));
        return;
    }
    for (int64_t b = 0; b < K / 16; ++b) {
        uint8_t c6[16], c4[16], s6, s4;
        float e6, e4;
        const uint8_t* cbest = c6;
        uint8_t sbest;
        nvfp4_block_candidate(x + 16 * b, t, 6.0f, c6, &s6, &e6);
        sbest = s6;
        if (four_six) {
            nvfp4_block_candidate(x + 16 * b, t, 4.0f, c4, &s4, &e4);
            if (e4 < e6) { cbest = c4; sbest = s4; }
        }
        sf[b] = sbest;
        for (int i = 0; i < 8; ++i)
            codes[8 * b + i] = (uint8_t)((cbest[2 * i] & 0xFu) | ((cbest[2 * i + 1] & 0xFu) << 4));
    }
}

static float nvfp4_scale_from_amax(float amax) { return amax / 2688.0f; }

/* One candidate of the 4/6 choice, exposed so tests can recompute both
 * candidates' errors independently: unpacked codes (16), SF byte, fp32 SSE. */
EXPORT void bsqo_nvfp4_block_candidate(const float* x16, float t, float mult,
                                       uint8_t* code16, uint8_t* sf, float* sse)
{
    nvfp4_block_candidate(x16, t, mult, code16, sf, sse);
}

/* Per-token (per-row) scales: the activation path. */
EXPORT void bsqo_nvfp4_quantize_rows(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx,
                                     int four_six, uint8_t* codes, uint8_t* sf, float* t)
{
    float* xf = (float*)malloc(sizeof(float) * (size_t)K);
    for (int64_t r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            xf[k] = bf16_to_f32(x[r * ldx + k]);
            amax = fmaxf(amax, fabsf(xf[k]));
        }
        t[r] = nvfp4_scale_from_amax(amax);
        nvfp4_row_given_t(xf, K, t[r], four_six, codes + r * (K / 2), sf + r * (K / 16));
    }
    free(xf);
}

/* Rows of binary32 values with caller-supplied second-level scales. */
EXPORT void bsqo_nvfp4_quantize_rows_given_t(const float* x, int64_t rows, int64_t K,
                                             const float* t, int four_six,
                                             uint8_t* codes, uint8_t* sf)
{
    for (int64_t r = 0; r < rows; ++r)
        nvfp4_row_given_t(x + r * K, K, t[r], four_six, codes + r * (K / 2), sf + r * (K / 16));
}

/* One scale per group of rows: the per-expert weight path (x is
 * [groups][rows][K]; for gate/up weights the rows of gate and up are
 * concatenated, so both share one scale, [MILES-IT] "Un quantizzatore
 * condiviso ...": gate and up are quantized together).  No 4/6 on weights. */
EXPORT void bsqo_nvfp4_quantize_group(const uint16_t* x, int64_t groups, int64_t rows, int64_t K,
                                      uint8_t* codes, uint8_t* sf, float* t)
{
    float* xf = (float*)malloc(sizeof(float) * (size_t)K);
    for (int64_t g = 0; g < groups; ++g) {
        const uint16_t* xg = x + g * rows * K;
        float amax = 0.0f;
        for (int64_t i = 0; i < rows * K; ++i) amax = fmaxf(amax, fabsf(bf16_to_f32(xg[i])));
        t[g] = nvfp4_scale_from_amax(amax);
        for (int64_t r = 0; r < rows; ++r) {
            for (int64_t k = 0; k < K; ++k) xf[k] = bf16_to_f32(xg[r * K + k]);
            int64_t row = g * rows + r;
            nvfp4_row_given_t(xf, K, t[g], 0, codes + row * (K / 2), sf + row * (K / 16));
        }
    }
    free(xf);
}

/* ------------------------------------------------------------------------
 * 2-D NVFP4: one E4M3 scale per 16 x 16 square block.  [TML-ZH] "第二个决定":
 * the alternative NVIDIA offers to requantizing in the backward pass is
 * square 16 x 16 block scaling, whose scale factors are the same before and
 * after the transpose; with 256 values under one scale a single large value
 * pushes the other 255 to zero, which is why the page's authors took the
 * dequantize-transpose-requantize route instead.
 * READING: the outer FP32 scale must not change under the transpose either,
 * so it is one per tensor, t = rn(amax / 2688) over the whole tensor (as for
 * weights); each tile then follows steps 3-4 of the per-row recipe with the
 * tile's amax in place of the 16-block's.  If t == 0 every code and scale is
 * 0.  Outputs: codes [rows][K/2] (the row-major packing of the 1 x 16
 * layout, low nibble = even column) and tile scales [rows/16][K/16].
 * rows % 16 == 0, K % 16 == 0.
 * ---------------------------------------------------------------------- */
EXPORT void bsqo_nvfp4_quantize_2d(const uint16_t* x, int64_t rows, int64_t K,
                                   uint8_t* codes, uint8_t* sf_tiles, float* t_out)
{
    if (rows <= 0 || K <= 0) {
        *t_out = 0.0f;
        return;
    }
    float amax = 0.0f;
    for (int64_t i = 0; i < rows * K; ++i) amax = fmaxf(amax, fabsf(bf16_to_f32(x[i])));
    const float t = nvfp4_scale_from_amax(amax);
    *t_out = t;
    memset(codes, 0, (size_t)(rows * K / 2));
    memset(sf_tiles, 0, (size_t)((rows / 16) * (K / 16)));
    if (t == 0.0f) return;
    for (int64_t tr = 0; tr < rows / 16; ++tr)
        for (int64_t tc = 0; tc < K / 16; ++tc) {
            float amax_t = 0.0f;
            for (int i = 0; i < 16; ++i)
                for (int j = 0; j < 16; ++j)
                    amax_t = fmaxf(amax_t, fabsf(bf16_to_f32(x[(16 * tr + i) * K + 16 * tc + j])));
            const float denom = 6.0f * t;
            const uint32_t sf = bsqo_e4m3_encode(amax_t / denom);
            const float d = bsqo_e4m3_decode(sf) * t;
            float enc = (d == 0.0f) ? 0.0f : 1.0f / d;
            if (isinf(enc)) enc = FLT_MAX;
            sf_tiles[tr * (K / 16) + tc] = (uint8_t)sf;
            for (int i = 0; i < 16; ++i)
                for (int j = 0; j < 16; ++j) {
                    const int64_t r = 16 * tr + i, k = 16 * tc + j;
                    const uint32_t code = bsqo_e2m1_encode(bf16_to_f32(x[r * K + k]) * enc);
                    codes[r * (K / 2) + k / 2] |= (uint8_t)((k & 1) ? (code << 4) : code);
                }
        }
}

/* ------------------------------------------------------------------------
 * 32-point random Hadamard transform before quantization.  [TML-ZH]
 * "第三个决定": a 32-dimensional random Hadamard transform spreads outliers
 * over their group before the values are block-quantized.
 * READINGS: per group of 32 consecutive elements of a row,
 * y = H32 (s . x), H32 the Sylvester Hadamard matrix (entries +-1,
 * H[i][j] = (-1)^popcount(i & j)), unnormalized: the per-token FP32 scale
 * absorbs the constant and H32 H32 = 32 I inverts it exactly.  Binary32,
 * by the butterfly h = 1, 2, 4, 8, 16 over pairs (i, i + h) with
 * (i & h) == 0: (v_i, v_{i+h}) <- (v_i + v_{i+h}, v_i - v_{i+h}).
 * s: one sign vector per tensor, s_j = -1 iff bit j of word 0 of
 * Philox4x32-10(key = seed, counter = (0, 0, 2, 0)) (stream 2: streams 0 and
 * 1 feed stochastic rounding).  The transformed rows are quantized with the
 * per-row recipe above (no 4/6); the pages' own target format for the
 * transformed values is not defined, so NVFP4 stands in.
 * ---------------------------------------------------------------------- */
EXPORT uint32_t bsqo_rht_signs(uint64_t seed)
{
    uint32_t ctr[4] = {0u, 0u, 2u, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    bsqo_philox4x32_10(ctr, key, out);
    return out[0];
}

EXPORT void bsqo_rht32(const float* x, int64_t n, uint32_t signs, float* y)
{
    for (int64_t g = 0; g + 32 <= n; g += 32) {
        float v[32];
        for (int j = 0; j < 32; ++j) v[j] = ((signs >> j) & 1u) ? -x[g + j] : x[g + j];
        for (int h = 1; h < 32; h <<= 1)
            for (int i = 0; i < 32; ++i)
                if ((i & h) == 0) {
                    const float a = v[i], b = v[i + h];
                    v[i] = a + b;
                    v[i + h] = a - b;
                }
        for (int j = 0; j < 32; ++j) y[g + j] = v[j];
    }
}

EXPORT void bsqo_nvfp4_quantize_rht(const uint16_t* x, int64_t rows, int64_t K, uint64_t seed,
                                    uint8_t* codes, uint8_t* sf, float* t)
{
    if (rows <= 0 || K <= 0) return;
    const uint32_t signs = bsqo_rht_signs(seed);
    float* xf = (float*)malloc(sizeof(float) * (size_t)K);
    float* y = (float*)malloc(sizeof(float) * (size_t)K);
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t k = 0; k < K; ++k) xf[k] = bf16_to_f32(x[r * K + k]);
        bsqo_rht32(xf, K, signs, y);
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) amax = fmaxf(amax, fabsf(y[k]));
        t[r] = nvfp4_scale_from_amax(amax);
        nvfp4_row_given_t(y, K, t[r], 0, codes + r * (K / 2), sf + r * (K / 16));
    }
    free(xf);
    free(y);
}

/* Step 5 above: binary32 dequantization of an NVFP4 tensor (per-row t). */
EXPORT void bsqo_nvfp4_dequantize(const uint8_t* codes, const uint8_t* sf, const float* t,
                                  int64_t rows, int64_t K, float* out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = codes[r * (K / 2) + k / 2];
            uint32_t code = (k & 1) ? (uint32_t)(byte >> 4) : (uint32_t)(byte & 0xFu);
            float s = bsqo_e4m3_decode(sf[r * (K / 16) + k / 16]);
            out[r * K + k] = (bsqo_e2m1_decode(code) * s) * t[r];
        }
}

/* The tensor-core scale-factor layout: the SF matrix [rows][K/16] is cut
 * into tiles of 128 rows x 4 SF (one 64-element K step); tiles are stored
 * row-tile major, K-tile minor, 512 bytes each, and inside a tile the SF of
 * (row r, column c) sits at (r % 32) * 16 + (r / 32) * 4 + c.  This is the
 * layout the block-scaled tensor-core MMA copies into tensor memory, 32 rows
 * of 16 bytes at a time; rows are padded to 128 and K to 64. */
EXPORT int64_t bsqo_sf_swizzled_offset(int64_t row, int64_t kblock, int64_t K)
{
    int64_t ktiles = (K + 63) / 64;
    int64_t tile = (row / 128) * ktiles + kblock / 4;
    int64_t r = row % 128;
    return tile * 512 + (r % 32) * 16 + (r / 32) * 4 + (kblock % 4);
}

/* Whole SF matrix [rows][cols] (cols = SF per row) into the layout above;
 * padding bytes are 0.  out holds ceil(rows/128)*128 * ceil(cols/4)*4 bytes. */
EXPORT void bsqo_sf_swizzle(const uint8_t* sf, int64_t rows, int64_t cols, uint8_t* out)
{
    int64_t rpad = (rows + 127) / 128 * 128, cpad = (cols + 3) / 4 * 4;
    memset(out, 0, (size_t)(rpad * cpad));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) out[bsqo_sf_swizzled_offset(r, c, 16 * cols)] = sf[r * cols + c];
}

/* ------------------------------------------------------------------------
 * MXFP8.  [LMSYS] "Recipe 1: End-to-end MXFP8": every 32 consecutive E4M3
 * values share one E8M0 scale, blocks are one-dimensional; TransformerEngine
 * materializes row-wise and column-wise copies, both from the original
 * high-precision input ([MILES-IT] "Un quantizzatore condiviso ...": blocks
 * must follow the reduction dimension).
 * READING (shared-exponent rule): X = clamp(floor(log2(amax_blk)) - 8,
 * -127, 127), SF byte = X + 127, code = E4M3(x * 2^-X) (the product is exact
 * wherever the code is not zero), so the largest element lands in [256, 512)
 * and saturates to 448 above it.  An all-zero block has SF 0 and codes 0.
 * The column copy is stored transposed: col_codes[K][rows], col_sf[K][rows/32].
 * ---------------------------------------------------------------------- */
static int mx_shared_exp(float amax)
{
    int e = ilogbf(amax);                    /* floor(log2(amax)), exact, subnormals too */
    int X = e - 8;
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    return X;
}

static void mx_block(const float* v, int64_t stride, uint8_t* codes, int64_t cstride,
                     uint8_t* sf, int sr, uint64_t seed, uint64_t idx0)
{
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i * stride]));
    if (amax == 0.0f) {
        *sf = 0;
        for (int i = 0; i < 32; ++i) codes[i * cstride] = 0;
        return;
    }
    int X = mx_shared_exp(amax);
    float mul = ldexpf(1.0f, -X);
    *sf = (uint8_t)(X + 127);
    for (int i = 0; i < 32; ++i) {
        float y = v[i * stride] * mul;
        codes[i * cstride] = (uint8_t)(sr ? bsqo_e4m3_encode_sr(y, bsqo_sr_bits16(seed, 1u, idx0 + (uint64_t)i))
                                          : bsqo_e4m3_encode(y));
    }
}

EXPORT void bsqo_mxfp8_quantize_rowcol(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx,
                                       uint8_t* row_codes, uint8_t* row_sf,
                                       uint8_t* col_codes, uint8_t* col_sf)
{
    float* xf = (float*)malloc(sizeof(float) * (size_t)(rows * K));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < K; ++k) xf[r * K + k] = bf16_to_f32(x[r * ldx + k]);
    if (row_codes)
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t b = 0; b < K / 32; ++b)
                mx_block(xf + r * K + 32 * b, 1, row_codes + r * K + 32 * b, 1,
                         row_sf + r * (K / 32) + b, 0, 0, 0);
    if (col_codes)
        for (int64_t k = 0; k < K; ++k)
            for (int64_t b = 0; b < rows / 32; ++b)
                mx_block(xf + (32 * b) * K + k, K, col_codes + k * rows + 32 * b, 1,
                         col_sf + k * (rows / 32) + b, 0, 0, 0);
    free(xf);
}

/* ------------------------------------------------------------------------
 * Backward requantization.  [TML-ZH] "第二个决定": the forward tensor uses
 * 1x16 row blocks; for the gradient GEMM it is transposed, so the same 16
 * values would fall into column groups with new scales.  The remedy taken:
 * dequantize the forward tensor to high precision, transpose, and quantize
 * again with stochastic rounding.
 * READINGS: D = dequant(input) in binary32 (step 5 above); Y = D^T; the
 * NVFP4 target quantizes each row of Y with the per-row recipe above (its
 * own t over the whole row, 6-candidate only); the MXFP8 target quantizes
 * each row of Y with the MXFP8 rule.  With sr != 0 the element codes use
 * stochastic rounding with bits bsqo_sr_bits16(seed, stream, idx), idx =
 * c * rows + r for the element (r, c) of D (its index in Y); stream 0 is the
 * NVFP4 target, 1 the MXFP8 target.  Scales are always RNE.
 * ---------------------------------------------------------------------- */
EXPORT void bsqo_requant_transpose(const uint8_t* codes, const uint8_t* sf, const float* t,
                                   int64_t rows, int64_t K, int sr, uint64_t seed,
                                   uint8_t* nv_codes_T, uint8_t* nv_sf_T, float* nv_t_T,
                                   uint8_t* mx_codes_T, uint8_t* mx_sf_T)
{
    int64_t M = rows;
    float* D = (float*)malloc(sizeof(float) * (size_t)(M * K));
    float* y = (float*)malloc(sizeof(float) * (size_t)M);
    bsqo_nvfp4_dequantize(codes, sf, t, M, K, D);
    for (int64_t c = 0; c < K; ++c) {
        float amax = 0.0f;
        for (int64_t r = 0; r < M; ++r) {
            y[r] = D[r * K + c];
            amax = fmaxf(amax, fabsf(y[r]));
        }
        uint64_t idx0 = (uint64_t)c * (uint64_t)M;
        if (nv_codes_T) {
            float tc = nvfp4_scale_from_amax(amax);
            nv_t_T[c] = tc;
            uint8_t* crow = nv_codes_T + c * (M / 2);
            uint8_t* srow = nv_sf_T + c * (M / 16);
            if (tc == 0.0f) {
                memset(crow, 0, (size_t)(M / 2));
                memset(srow, 0, (size_t)(M / 16));
            } else {
                for (int64_t b = 0; b < M / 16; ++b) {
                    const float* xb = y + 16 * b;
                    float amax_b = 0.0f;
                    for (int i = 0; i < 16; ++i) amax_b = fmaxf(amax_b, fabsf(xb[i]));
                    float denom = 6.0f * tc;
                    uint32_t s = bsqo_e4m3_encode(amax_b / denom);
                    float d = bsqo_e4m3_decode(s) * tc;
                    float enc = (d == 0.0f) ? 0.0f : 1.0f / d;
                    if (isinf(enc)) enc = FLT_MAX;
                    srow[b] = (uint8_t)s;
                    for (int i = 0; i < 16; i += 2) {
                        uint32_t cc[2];
                        for (int h = 0; h < 2; ++h) {
                            float q = xb[i + h] * enc;
                            uint64_t idx = idx0 + (uint64_t)(16 * b + i + h);
                            cc[h] = sr ? bsqo_e2m1_encode_sr(q, bsqo_sr_bits16(seed, 0u, idx))
                                       : bsqo_e2m1_encode(q);
                        }
                        crow[8 * b + i / 2] = (uint8_t)((cc[0] & 0xFu) | ((cc[1] & 0xFu) << 4));
                    }
                }
            }
        }
        if (mx_codes_T)
            for (int64_t b = 0; b < M / 32; ++b)
                mx_block(y + 32 * b, 1, mx_codes_T + c * M + 32 * b, 1, mx_sf_T + c * (M / 32) + b,
                         sr, seed, idx0 + (uint64_t)(32 * b));
    }
    free(y);
    free(D);
}

/* ------------------------------------------------------------------------
 * Block-scaled GEMM.  [LMSYS] "Why Blackwell changes the math": the tensor
 * cores apply the per-block scales in hardware; "Results": the per-token
 * FP32 scale belongs in the GEMM epilogue.  The plain definition: both
 * operands dequantized exactly (value * block scale * FP32 scale is exact in
 * fp64), out[m][n] = sum_k A[m][k] * B[n][k] in fp64, k ascending.
 * abs_out (optional) receives sum_k |A[m][k] * B[n][k]| for tolerances.
 * ---------------------------------------------------------------------- */
static double deq64(const uint8_t* codes, const uint8_t* sf, int64_t row, int64_t k, int64_t K)
{
    uint8_t byte = codes[row * (K / 2) + k / 2];
    uint32_t code = (k & 1) ? (uint32_t)(byte >> 4) : (uint32_t)(byte & 0xFu);
    return (double)bsqo_e2m1_decode(code) * (double)bsqo_e4m3_decode(sf[row * (K / 16) + k / 16]);
}

EXPORT void bsqo_gemm_nvfp4(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_t,
                            int64_t M, int64_t K,
                            const uint8_t* b_codes, const uint8_t* b_sf, float b_t, int64_t N,
                            double* out, double* abs_out)
{
    double* bd = (double*)malloc(sizeof(double) * (size_t)(N * K));
    double* ad = (double*)malloc(sizeof(double) * (size_t)K);
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) bd[n * K + k] = deq64(b_codes, b_sf, n, k, K) * (double)b_t;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t k = 0; k < K; ++k) ad[k] = deq64(a_codes, a_sf, m, k, K) * (double)a_t[m];
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = ad[k] * bd[n * K + k];
                acc += p;
                aacc += fabs(p);
            }
            out[m * N + n] = acc;
            if (abs_out) abs_out[m * N + n] = aacc;
        }
    }
    free(ad);
    free(bd);
}

/* GEMM on exactly dequantized MXFP8 operands (fp64): out[m][n] =
 * sum_k A[m][k] B[n][k], A and B K-major, each element E4M3(code) *
 * 2^(E8M0(sf of its 32-block) - 127) ([MILES-IT] "Il supporto Miles ...":
 * the MXFP8 recipe also runs the weight- and data-gradient GEMMs in MXFP8;
 * [LMSYS] "Recipe 1: End-to-end MXFP8").  a_t / b_t (FP32) multiply the rows
 * of A and all of B (1 for plain MXFP8).  SF linear [rows][K/32]. */
static double mx_deq64(const uint8_t* codes, const uint8_t* sf, int64_t r, int64_t k, int64_t K)
{
    return (double)bsqo_e4m3_decode(codes[r * K + k]) * (double)bsqo_e8m0_decode(sf[r * (K / 32) + k / 32]);
}

EXPORT void bsqo_gemm_mxfp8(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_t, int64_t M, int64_t K,
                            const uint8_t* b_codes, const uint8_t* b_sf, float b_t, int64_t N,
                            double* out, double* abs_out)
{
    double* bd = (double*)malloc(sizeof(double) * (size_t)(N * K));
    double* ad = (double*)malloc(sizeof(double) * (size_t)K);
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) bd[n * K + k] = mx_deq64(b_codes, b_sf, n, k, K) * (double)b_t;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t k = 0; k < K; ++k) ad[k] = mx_deq64(a_codes, a_sf, m, k, K) * (double)a_t[m];
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double p = ad[k] * bd[n * K + k];
                acc += p;
                aacc += fabs(p);
            }
            out[m * N + n] = acc;
            if (abs_out) abs_out[m * N + n] = aacc;
        }
    }
    free(ad);
    free(bd);
}

/* One output element per sample: row a_rows[s] of A against row b_rows[s]
 * of B (B rows of all groups stacked), with B's FP32 scale b_t[b_group[s]]. */
EXPORT void bsqo_gemm_nvfp4_sampled(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_t,
                                    int64_t K,
                                    const uint8_t* b_codes, const uint8_t* b_sf, const float* b_t,
                                    const int64_t* a_rows, const int64_t* b_rows,
                                    const int64_t* b_group, int64_t n_samples,
                                    double* out, double* abs_out)
{
    for (int64_t s = 0; s < n_samples; ++s) {
        int64_t m = a_rows[s], n = b_rows[s];
        double ta = (double)a_t[m], tb = (double)b_t[b_group[s]];
        double acc = 0.0, aacc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = (deq64(a_codes, a_sf, m, k, K) * ta) * (deq64(b_codes, b_sf, n, k, K) * tb);
            acc += p;
            aacc += fabs(p);
        }
        out[s] = acc;
        if (abs_out) abs_out[s] = aacc;
    }
}

/* ------------------------------------------------------------------------
 * MoE expert forward pieces.
 * Dispatch ([TML-ZH] "第三个决定": tokens travel to their experts already
 * quantized).  READING: routed rows are grouped by expert, each expert's
 * segment padded to a multiple of `pad` rows; inside a segment rows are in
 * ascending (token, k) order.  offsets[E+1] are the padded segment starts,
 * slot_of[t*k + j] the row of routed pair (t, j), row_src[row] = t*k + j or
 * -1 for padding.  Returns the padded row count.
 * ---------------------------------------------------------------------- */
EXPORT int64_t bsqo_route(const int32_t* topk_ids, int64_t T, int64_t k, int64_t E, int64_t pad,
                          int32_t* offsets, int32_t* slot_of, int32_t* row_src)
{
    int64_t* count = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    for (int64_t i = 0; i < T * k; ++i) count[topk_ids[i]]++;
    int64_t off = 0;
    for (int64_t e = 0; e < E; ++e) {
        offsets[e] = (int32_t)off;
        off += (count[e] + pad - 1) / pad * pad;
    }
    offsets[E] = (int32_t)off;
    if (row_src)
        for (int64_t r = 0; r < off; ++r) row_src[r] = -1;
    int64_t* fill = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    for (int64_t i = 0; i < T * k; ++i) {           /* ascending (token, k) */
        int64_t e = topk_ids[i];
        int64_t row = offsets[e] + fill[e]++;
        slot_of[i] = (int32_t)row;
        if (row_src) row_src[row] = (int32_t)i;
    }
    free(fill);
    free(count);
    return off;
}

/* [MILES-IT] "Un quantizzatore condiviso ...": SwiGLU experts run gate and up
 * as one fused matmul.  READING: columns [0, I) are gate, [I, 2I) are up;
 * h = silu(gate) * up with silu(g) = g / (1 + exp(-g)), all in fp64. */
EXPORT void bsqo_swiglu(const double* gate_up, int64_t rows, int64_t I, double* h)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < I; ++j) {
            double g = gate_up[r * 2 * I + j], u = gate_up[r * 2 * I + I + j];
            h[r * I + j] = (g / (1.0 + exp(-g))) * u;
        }
}

/* Round an fp64 value to the nearest bf16 (ties to even), directly from fp64
 * so there is no double rounding. */
EXPORT uint16_t bsqo_f64_to_bf16(double v)
{
    if (isnan(v)) return 0x7FC0u;
    double a = fabs(v);
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double r;
    if (a == 0.0) return sign;
    if (a < ldexp(1.0, -126)) {
        r = nearbyint(a * ldexp(1.0, 133)) * ldexp(1.0, -133);   /* subnormal grid 2^-133 */
    } else {
        int e;
        double m = frexp(a, &e);                 /* a = m * 2^e, m in [0.5, 1) */
        r = ldexp(nearbyint(ldexp(m, 8)), e - 8);  /* 8 significant bits */
    }
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);  /* overflow to inf */
    float f = (float)r;                           /* exact: r has <= 8 significant bits */
    return (uint16_t)(sign | (f32_to_bits(f) >> 16));
}

EXPORT void bsqo_f64_to_bf16_array(const double* v, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = bsqo_f64_to_bf16(v[i]);
}

/* Combine: y[t] = bf16( sum_{j < k} w[t][j] * out[slot_of[t*k + j]] ), fp64,
 * j ascending.  out_rows are the per-routed-row expert outputs (bf16). */
EXPORT void bsqo_combine(const uint16_t* out_rows, int64_t H, const int32_t* slot_of,
                         const float* topk_w, int64_t T, int64_t k, uint16_t* y)
{
    for (int64_t t = 0; t < T; ++t)
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int64_t j = 0; j < k; ++j) {
                int64_t row = slot_of[t * k + j];
                acc += (double)topk_w[t * k + j] * (double)bf16_to_f32(out_rows[row * H + h]);
            }
            y[t * H + h] = bsqo_f64_to_bf16(acc);
        }
}
