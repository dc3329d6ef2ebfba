// requant.cu -- the backward requantization ("End-to-End 4-Bit Training",
// "第二个决定": dequantize the forward NVFP4 tensor, transpose it, quantize it
// again with stochastic rounding), to NVFP4 and/or MXFP8, with round-to-nearest
// as an option, plus the allocation-free variant of the call.
//
// Two kernels.  k_rq_colmax reads the input once and folds the column maxima
// of |D| (D the dequantized input) into a K-word array: the NVFP4 target's
// per-row FP32 scale of Y = D^T needs the maximum over a whole row of Y, i.e.
// over every source row.  k_rq_tile then dequantizes 256 x 64 source tiles
// into shared memory, transposed, and encodes the tile's 64 output rows.
//
// Both are bound by instruction issue, not by HBM (the input is 0.56 byte an
// element, the two outputs 1.6), so the arithmetic is laid out for few
// instructions an element:
//   - dequantization works on f16 pairs: E2M1 code pairs to f16x2 with the
//     hardware conversion, one packed multiply by the E4M3 scale pair (exact:
//     both are f16 values with a product of at most 6 significant bits), then
//     one conversion to binary32 and one multiply by the row scale per value;
//   - the tile is staged as f16x2 pairs of neighbouring source rows (16 KB of
//     a 256 x 64 tile per 32 columns), so the transposition costs one 4-byte
//     shared store per two values;
//   - the stochastic encoders have no branch and no float-to-integer
//     conversion (see sr_t24).
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace bsq {
namespace {

// ---------------------------------------------------------------------------
// Stochastic rounding with 16 random bits r (the rule of quantize_nvfp4 and
// quantize_mxfp8 targets: with lo <= |v| < hi the neighbouring grid points,
// round up iff r < 65536 (|v| - lo) / (hi - lo), saturate at the largest
// finite value).
//
// Both formats have a normal range where the grid keeps the top bits of the
// binary32 significand (E2M1: 1 bit on [1, 6]; E4M3: 3 bits on [2^-6, 448])
// and a uniform grid below it with the spacing of the lowest normal binade
// (E2M1: 0.5 on [0, 1); E4M3: 2^-9 on [0, 2^-6)).  The value is first scaled
// by a power of two, exactly, so that the normal range becomes [4, S] (E2M1:
// x 4; E4M3: x 256) and saturated at S.  Below 4, s / 2 + 2 maps [0, 4) onto
// the binade [2, 4) with the same relative grid as the uniform one, and the
// rounding up of that sum (fma.rp) keeps, exactly, whether any bit of s
// below the binary32 grid of [2, 4) is set: for an integer comparison
// against r, ceil() of the dropped fraction decides the same way as the
// exact fraction.  On [4, S], s / 2 + 2 <= s; on [0, 4), s / 2 + 2 > s, so
// z = max(s, s / 2 + 2 rounded up) is the operand of the integer rounding
// in both ranges.
//
// z lies in [2, 2^17), whose binary32 exponents are 128 .. 143: shifting its
// bit pattern left by 4 (E4M3) or 2 (E2M1) drops the constant exponent bits
// and leaves the code magnitude in bits 24 .. 30 (E4M3: the low 4 exponent
// bits and 3 significand bits, which is the E4M3 code with its bias of 7; E2M1:
// the low 2 exponent bits and 1 significand bit, bits 24 .. 26) above 24
// dropped bits.  Adding 2^24 - 1 - (r << 8) carries into bit 24 iff the
// dropped bits exceed r << 8, i.e. iff the dropped fraction exceeds r / 2^16:
// the rule above.  The code is byte 3 of the sum; the sign is bit 7 of byte 3
// of the input.
// ---------------------------------------------------------------------------

// r << 8 for the 16-bit draw in the low (h = 0) or high (h = 1) half of w.
BSQ_DEVICE uint32_t sr_r8(uint32_t w, int h) { return __byte_perm(w, 0u, h ? 0x4324u : 0x4104u); }

template <int SHIFT>
BSQ_DEVICE uint32_t sr_t24(float s, uint32_t r8)
{
    const float z = fmaxf(s, __fmaf_ru(s, 0.5f, 2.0f));
    return (__float_as_uint(z) << SHIFT) + (0xFFFFFFu - r8);
}

// Byte 3 of four words, as bytes 0..3 of one word.
BSQ_DEVICE uint32_t byte3x4(uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    return __byte_perm(__byte_perm(a, b, 0x7373u), __byte_perm(c, d, 0x7373u), 0x5410u);
}

// Four binary32 values (already multiplied by the block's 2^-X) -> four E4M3
// bytes with stochastic rounding; draws: x0, x1 from the halves of wa, x2, x3
// from those of wb.
BSQ_DEVICE uint32_t e4m3x4_sr(float x0, float x1, float x2, float x3, uint32_t wa, uint32_t wb)
{
    const uint32_t t0 = sr_t24<4>(fminf(fabsf(x0) * 256.0f, 114688.0f), sr_r8(wa, 0));
    const uint32_t t1 = sr_t24<4>(fminf(fabsf(x1) * 256.0f, 114688.0f), sr_r8(wa, 1));
    const uint32_t t2 = sr_t24<4>(fminf(fabsf(x2) * 256.0f, 114688.0f), sr_r8(wb, 0));
    const uint32_t t3 = sr_t24<4>(fminf(fabsf(x3) * 256.0f, 114688.0f), sr_r8(wb, 1));
    const uint32_t sg = byte3x4(__float_as_uint(x0), __float_as_uint(x1), __float_as_uint(x2), __float_as_uint(x3));
    return byte3x4(t0, t1, t2, t3) | (sg & 0x80808080u);
}

// Eight binary32 values (already multiplied by the block's encode scale) ->
// eight E2M1 codes (element i in nibble i) with stochastic rounding; the
// draws of element i are half i & 1 of word i >> 1 of rb.
BSQ_DEVICE uint32_t e2m1x8_sr(const float (&x)[8], const uint4& rb)
{
    const uint32_t w[4] = {rb.x, rb.y, rb.z, rb.w};
    uint32_t t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) t[i] = sr_t24<2>(fminf(fabsf(x[i]) * 4.0f, 24.0f), sr_r8(w[i >> 1], i & 1));
    const uint32_t ca = byte3x4(t[0], t[1], t[2], t[3]), cb = byte3x4(t[4], t[5], t[6], t[7]);
    const uint32_t sa = byte3x4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                                __float_as_uint(x[3]));
    const uint32_t sb = byte3x4(__float_as_uint(x[4]), __float_as_uint(x[5]), __float_as_uint(x[6]),
                                __float_as_uint(x[7]));
    const uint32_t na = ca | ((sa >> 4) & 0x08080808u), nb = cb | ((sb >> 4) & 0x08080808u);
    return __byte_perm(na | (na >> 4), nb | (nb >> 4), 0x6420u);  // nibbles 2i, 2i+1 from bytes 2i, 2i+1
}

// Philox draws of 8 consecutive elements 8 g .. 8 g + 7 of one target; below
// 2^35 elements (not WIDE) the counter's second word is 0 at compile time.
template <uint32_t STREAM, bool WIDE>
BSQ_DEVICE uint4 sr_bits(const PhiloxKeys& k, uint64_t g)
{
    return philox4x32_10_keys(make_uint4((uint32_t)g, WIDE ? (uint32_t)(g >> 32) : 0u, STREAM, 0u), k);
}

// f16x2 pair -> two binary32 values times (t0, t1), each rounded once.
BSQ_DEVICE void h2_times(uint32_t h2, float t0, float t1, float& a, float& b)
{
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
    a = __fmul_rn(f.x, t0);
    b = __fmul_rn(f.y, t1);
}

// The four bytes of w (two E2M1 codes each, low nibble first) -> four f16x2.
BSQ_DEVICE void e2m1x8_f16x2(uint32_t w, uint32_t (&h)[4])
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

// rn(1 / m) for e4m3_of_quotient, or 0 where that quotient is to be taken
// exactly: m zero or non-finite, or a reciprocal outside the normal range
// (there its relative error is not bounded by one unit in the last place).
BSQ_DEVICE float quotient_inv(float m)
{
    const float r = __frcp_rn(m);
    return (r >= 1.17549435e-38f && r <= kFltMax) ? r : 0.0f;
}

// The NVFP4 block scale E4M3(rn(a / m)) (RNE, satfinite; a = the block's
// amax, m = rn(6 t)) given inv = quotient_inv(m).  q = rn(a * inv) lies
// within 1.5 units in the last place of a / m, so when q (1 - 2^-20) and
// q (1 + 2^-20) encode to the same byte -- E4M3 rounding is monotone -- so
// does the correctly rounded quotient; otherwise (q near an E4M3 rounding
// boundary, or inv = 0) the quotient is computed exactly.  Here the divisor
// changes with every output row, so a division per block would not be
// hoisted; this costs one multiply, two scalings and one conversion in all
// but a few blocks in 10^5.
BSQ_DEVICE uint32_t e4m3_of_quotient(float a, float m, float inv)
{
    const float q = __fmul_rn(a, inv);
    uint32_t two;
    asm("{\n\t.reg .b16 b;\n\tcvt.rn.satfinite.e4m3x2.f32 b, %1, %2;\n\tcvt.u32.u16 %0, b;\n\t}"
        : "=r"(two)
        : "f"(__fmul_rn(q, 1.00000095367431640625f)), "f"(__fmul_rn(q, 0.99999904632568359375f)));
    if (inv != 0.0f && (two & 0xFFu) == (two >> 8)) return two & 0xFFu;
    return e4m3_rn(__fdiv_rn(a, m));
}

// Two E4M3 bytes (low = first) -> f16x2.
BSQ_DEVICE uint32_t e4m3x2_f16x2(uint32_t two)
{
    uint32_t h;
    asm("{\n\t.reg .b16 b;\n\tcvt.u16.u32 b, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, b;\n\t}" : "=r"(h) : "r"(two));
    return h;
}

BSQ_DEVICE float f16lo_to_f32(uint32_t h2)
{
    return __low2float(*reinterpret_cast<const __half2*>(&h2));
}

BSQ_DEVICE uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// SF byte of 16-column block b of row r.
template <bool SWZ>
BSQ_DEVICE const uint8_t* sf_at(const uint8_t* sf, int64_t r, int64_t b, int64_t nsf)
{
    return sf + (SWZ ? sf_swizzled(r, b, (nsf + 3) >> 2) : r * nsf + b);
}

// ---------------------------------------------------------------------------
// Column maxima of |D|, D = rn(rn(e2m1 * sf) * t).  Persistent: CTA (x, y)
// of a grid of about four CTAs per SM (64 registers: 32 warps an SM to hide
// the load latency) owns the 512 columns of chunk x (lane l the 16 columns of
// block 32 x + l: one 8-byte code load and one SF byte per row) and, per
// warp, batches of 8 consecutive rows (batch y * 8 + warp, then every 8 G-th,
// G = gridDim.y).  A batch's 24 loads are all in flight at once, then folded
// (3-input max, two rows per step); 8 rows from a multiple of 8 share one SF
// address computation (in the swizzled layout they sit in one 32-row group,
// 16 bytes apart).  Double-buffering the batches in registers (128 registers,
// 2 CTAs an SM) was slower.  The 8 warps' maxima are folded in shared memory
// and each column's maximum goes to colmax with one unsigned atomicMax on the
// bits of a non-negative float (order-independent, so deterministic).  colmax
// must hold zeros beforehand.
constexpr int CM_COLS = 512;

BSQ_DEVICE void cm_row(uint2 w, uint32_t sfb, float t, float (&d)[16])
{
    const uint32_t s2 = e4m3x2_f16x2(sfb * 0x101u);
    const uint32_t ww[2] = {w.x & 0x77777777u, w.y & 0x77777777u};  // |codes|
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        uint32_t h[4];
        e2m1x8_f16x2(ww[q], h);
#pragma unroll
        for (int i = 0; i < 4; ++i) h2_times(hmul2(h[i], s2), t, t, d[8 * q + 2 * i], d[8 * q + 2 * i + 1]);
    }
}

struct CmBatch {  // one warp-batch of 8 rows: codes, SF bytes, row scales
    uint2 w[8];
    uint32_t s[8];
    float t[8];
};

template <bool SWZ>
BSQ_DEVICE bool cm_load(CmBatch& B, const uint8_t* codes, const uint8_t* sf, const float* row_scale, int64_t batch,
                        int64_t nbatch, int64_t b, int64_t nsf, int64_t ldc)
{
    if (batch >= nbatch) return false;
    const int64_t rb = 8 * batch;  // rows rb .. rb + 7, all in range (rows % 8 == 0)
    const uint8_t* cp = codes + rb * ldc + 8 * b;
    const uint8_t* sp = sf_at<SWZ>(sf, rb, b, nsf);
    const int64_t sstep = SWZ ? 16 : nsf;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        B.w[u] = __ldg(reinterpret_cast<const uint2*>(cp + u * ldc));
        B.s[u] = __ldg(sp + u * sstep);
        B.t[u] = __ldg(row_scale + rb + u);
    }
    return true;
}

BSQ_DEVICE void cm_fold(const CmBatch& B, float (&acc)[16])
{
#pragma unroll
    for (int u = 0; u < 8; u += 2) {
        float da[16], db[16];
        cm_row(B.w[u], B.s[u], B.t[u], da);
        cm_row(B.w[u + 1], B.s[u + 1], B.t[u + 1], db);
#pragma unroll
        for (int j = 0; j < 16; ++j) asm("max.f32 %0, %0, %1, %2;" : "+f"(acc[j]) : "f"(da[j]), "f"(db[j]));
    }
}

template <bool SWZ>
__global__ void __launch_bounds__(256, 4) k_rq_colmax(const uint8_t* __restrict__ codes,
                                                      const uint8_t* __restrict__ sf,
                                                      const float* __restrict__ row_scale, int64_t rows, int64_t K,
                                                      unsigned int* __restrict__ colmax)
{
    pdl_enter();
    __shared__ float red[8][32][17];  // [warp][lane][column of the lane's block], padded
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t b = (int64_t)blockIdx.x * (CM_COLS / 16) + lane;  // this lane's 16-column block
    const int64_t nsf = K >> 4, ldc = K >> 1, nbatch = rows >> 3;
    const int64_t step = 8 * (int64_t)gridDim.y;
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
    if (b < nsf) {
        CmBatch A;
        for (int64_t bi = (int64_t)blockIdx.y * 8 + warp; cm_load<SWZ>(A, codes, sf, row_scale, bi, nbatch, b, nsf, ldc);
             bi += step)
            cm_fold(A, acc);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) red[warp][lane][j] = acc[j];
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int c = threadIdx.x + 256 * h;  // column of the CTA's 512
        const int l = c >> 4, j = c & 15;
        float v = red[0][l][j];
#pragma unroll
        for (int w = 1; w < 8; ++w) v = fmaxf(v, red[w][l][j]);
        const int64_t gc = (int64_t)blockIdx.x * CM_COLS + c;
        if (gc < K && v > 0.0f) atomicMax(colmax + gc, __float_as_uint(v));
    }
}

// ---------------------------------------------------------------------------
// The tile pass.  CTA: 256 source rows (m) x 64 source columns (k), 256
// threads.
//
// Stage 1: thread (p, h) = (tid & 127, tid >> 7) dequantizes source rows
// 2p, 2p + 1 over columns 32 h .. 32 h + 31.  Interleaving the two rows'
// code words by nibble gives bytes that hold one column of both rows, which
// the E2M1 pair conversion turns into (row 2p, row 2p + 1) f16x2 values; one
// packed multiply by the two rows' E4M3 scales gives the exact products,
// stored as word p of row k of DT[64][128] (16-byte chunk c of a row at
// c ^ ((c >> 3) & 1), so the readers below hit distinct banks).  Rows past
// the input are staged as zeros (their outputs are not stored, and their
// scale bytes, stored where the swizzled layout pads, are 0).
//
// Stage 2: each half-warp produces one output row k (a source column) per
// step, warp w taking rows 16 i + 2 w + hh: lane l16 owns m = 16 l16 .. +15
// (one NVFP4 block, half of one MXFP8 block), converts its 8 pairs to
// binary32 and multiplies by its 16 row scales.  MXFP8: the block maximum
// with the neighbour lane, E8M0 exponent, 16 code bytes.  NVFP4: the row's
// FP32 scale from the column maximum, the block's E4M3 scale, 8 code bytes.
// Scale bytes are collected in shared memory and stored as 32-bit words
// after the tile.
constexpr int RT_M = 256, RT_K = 64;

BSQ_DEVICE int dt_word(int k, int p) { return k * (RT_M / 2) + (p ^ (((p >> 5) & 1) << 2)); }

template <bool SWZ, bool SR, bool NV, bool MX, bool WIDE>
__global__ void __launch_bounds__(256) k_rq_tile(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ sf,
                                                 const float* __restrict__ row_scale, int64_t rows, int64_t K,
                                                 const unsigned int* __restrict__ colmax,
                                                 uint8_t* __restrict__ nv_codes, uint8_t* __restrict__ nv_sf,
                                                 float* __restrict__ nv_scale, uint8_t* __restrict__ mx_codes,
                                                 uint8_t* __restrict__ mx_sf, const PhiloxKeys keys)
{
    pdl_enter();
    __shared__ __align__(16) uint32_t DT[RT_K * (RT_M / 2)];  // 32 KB
    __shared__ __align__(16) float tsrc[RT_M];
    __shared__ float4 tq[RT_K];  // (t, rn(6 t), quotient_inv(rn(6 t))) of the NVFP4 output rows
    __shared__ __align__(16) uint8_t sfo_nv[RT_K][RT_M / 16];
    __shared__ __align__(16) uint8_t sfo_mx[RT_K][RT_M / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t m0 = (int64_t)blockIdx.y * RT_M, k0 = (int64_t)blockIdx.x * RT_K;
    const int64_t nsf_in = K >> 4;
    {
        const int p = tid & (RT_M / 2 - 1), h = tid >> 7;
        const int64_t ga = m0 + 2 * p;              // rows ga, ga + 1 (rows is even)
        const int64_t kc = k0 + 32 * h;             // first column of this half
        const int64_t left = K - kc;                // K % 16 == 0: 0, 16 or >= 32 columns in range
        const int nblk = left >= 32 ? 2 : (left >= 16 ? 1 : 0);
        uint32_t a[4] = {0u, 0u, 0u, 0u}, bw[4] = {0u, 0u, 0u, 0u};
        uint32_t sa = 0u, sb = 0u;
        float ta = 0.0f, tb = 0.0f;
        if (ga < rows && nblk > 0) {
            const uint8_t* pa = codes + ga * (K >> 1) + (kc >> 1);
            const uint8_t* pb = pa + (K >> 1);
            if (nblk == 2 && (K & 31) == 0) {
                const uint4 x = __ldg(reinterpret_cast<const uint4*>(pa));
                const uint4 y = __ldg(reinterpret_cast<const uint4*>(pb));
                a[0] = x.x; a[1] = x.y; a[2] = x.z; a[3] = x.w;
                bw[0] = y.x; bw[1] = y.y; bw[2] = y.z; bw[3] = y.w;
            } else {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    if (q < nblk) {
                        const uint2 x = __ldg(reinterpret_cast<const uint2*>(pa) + q);
                        const uint2 y = __ldg(reinterpret_cast<const uint2*>(pb) + q);
                        a[2 * q] = x.x; a[2 * q + 1] = x.y;
                        bw[2 * q] = y.x; bw[2 * q + 1] = y.y;
                    }
                }
            }
            // blocks b0, b0 + 1 (b0 even) of rows ga, ga + 1 (ga even): adjacent
            // bytes, and the second row 16 bytes (swizzled: same 32-row group)
            // or one row further
            const int64_t b0 = kc >> 4;
            const uint8_t* s0 = sf_at<SWZ>(sf, ga, b0, nsf_in);
            const uint8_t* s1 = s0 + (SWZ ? 16 : nsf_in);
            sa = __ldg(s0);
            sb = __ldg(s1);
            if (nblk == 2) {
                sa |= (uint32_t)__ldg(s0 + 1) << 8;
                sb |= (uint32_t)__ldg(s1 + 1) << 8;
            }
            ta = __ldg(row_scale + ga);
            tb = __ldg(row_scale + ga + 1);
        }
        if (h == 0) {
            tsrc[2 * p] = ta;
            tsrc[2 * p + 1] = tb;
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint32_t s2 = e4m3x2_f16x2((sa >> (8 * q) & 0xFFu) | ((sb >> (8 * q) & 0xFFu) << 8));
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int j = 2 * q + jj;  // code word: columns 8 j .. 8 j + 7 of the half
                const uint32_t ev = (a[j] & 0x0F0F0F0Fu) | ((bw[j] << 4) & 0xF0F0F0F0u);
                const uint32_t od = ((a[j] >> 4) & 0x0F0F0F0Fu) | (bw[j] & 0xF0F0F0F0u);
                uint32_t he[4], ho[4];
                e2m1x8_f16x2(ev, he);
                e2m1x8_f16x2(od, ho);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int kk = 32 * h + 8 * j + 2 * i;
                    DT[dt_word(kk, p)] = hmul2(he[i], s2);
                    DT[dt_word(kk + 1, p)] = hmul2(ho[i], s2);
                }
            }
        }
        if (NV && tid < RT_K) {
            const int64_t gk = k0 + tid;
            float t = 0.0f;
            if (gk < K) {
                t = __fdiv_rn(__uint_as_float(__ldg(colmax + gk)), kNvfp4ScaleDivisor);
                if (blockIdx.y == 0) nv_scale[gk] = t;
            }
            const float six = __fmul_rn(6.0f, t);
            tq[tid] = make_float4(t, six, quotient_inv(six), 0.0f);
        }
    }
    __syncthreads();
    const int l16 = lane & 15, hh = lane >> 4;
    const int64_t gm = m0 + 16 * l16;  // first source row of this lane
    const bool valid = gm < rows;      // rows % 32 == 0: whole MXFP8 blocks drop out
    float tl[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float4 f = *reinterpret_cast<const float4*>(tsrc + 16 * l16 + 4 * j);
        tl[4 * j] = f.x; tl[4 * j + 1] = f.y; tl[4 * j + 2] = f.z; tl[4 * j + 3] = f.w;
    }
    const uint64_t g8 = ((uint64_t)(k0 + 2 * warp + hh) * (uint64_t)rows + (uint64_t)gm) >> 3;
    const uint64_t g8_step = 2ull * (uint64_t)rows;  // 16 output rows further
    // this lane's code bytes in its first output row (k0 + 2 warp + hh), and
    // the stride of 16 output rows
    uint8_t* mxp = MX ? mx_codes + (k0 + 2 * warp + hh) * rows + gm : nullptr;
    uint8_t* nvp = NV ? nv_codes + (k0 + 2 * warp + hh) * (rows >> 1) + (gm >> 1) : nullptr;
    const int64_t mx_step = 16 * rows, nv_step = 8 * rows;
    for (int it = 0; it < RT_K / 16; ++it) {
        if (k0 + 16 * it >= K) break;  // K % 16 == 0: the 16 rows of a step are all in or all out
        const int kk = 16 * it + 2 * warp + hh;
        float v[16];
        {
            const int c0 = 2 * l16;  // 16-byte chunks c0, c0 + 1 of row kk
            const int sw = (c0 >> 3) & 1;
            const uint4 lo = *reinterpret_cast<const uint4*>(DT + kk * (RT_M / 2) + 4 * (c0 ^ sw));
            const uint4 hi = *reinterpret_cast<const uint4*>(DT + kk * (RT_M / 2) + 4 * ((c0 + 1) ^ sw));
            const uint32_t hw[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) h2_times(hw[i], tl[2 * i], tl[2 * i + 1], v[2 * i], v[2 * i + 1]);
        }
        float am = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(v[i]));
        const uint64_t g = g8 + (uint64_t)it * g8_step;  // Philox counter of v[0..7]; v[8..15]: g + 1
        if (MX) {
            const float ab = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));  // MXFP8 block (32 rows)
            uint32_t w[4] = {0u, 0u, 0u, 0u}, sc = 0u;
            if (ab > 0.0f) {
                const int X = mx_exponent(__float_as_uint(ab));
                const float mul = mx_multiplier(X);
                sc = (uint32_t)(X + 127);
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) x[i] = __fmul_rn(v[i], mul);
                if (SR) {
#pragma unroll
                    for (int hb = 0; hb < 2; ++hb) {
                        const uint4 rb = sr_bits<1u, WIDE>(keys, g + hb);
                        w[2 * hb] = e4m3x4_sr(x[8 * hb], x[8 * hb + 1], x[8 * hb + 2], x[8 * hb + 3], rb.x, rb.y);
                        w[2 * hb + 1] = e4m3x4_sr(x[8 * hb + 4], x[8 * hb + 5], x[8 * hb + 6], x[8 * hb + 7], rb.z, rb.w);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) w[q] = e4m3x4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
                }
            }
            if (valid) *reinterpret_cast<uint4*>(mxp + it * mx_step) = make_uint4(w[0], w[1], w[2], w[3]);
            if ((l16 & 1) == 0) sfo_mx[kk][l16 >> 1] = (uint8_t)sc;
        }
        if (NV) {
            const float4 tt = tq[kk];
            uint32_t w[2] = {0u, 0u}, sfb = 0u;
            if (tt.x != 0.0f) {
                BlockScale bs;
                bs.sf = e4m3_of_quotient(am, tt.y, tt.z);
                bs.d = __fmul_rn(f16lo_to_f32(e4m3x2_f16x2(bs.sf)), tt.x);
                const float enc = bs.d == 0.0f ? 0.0f : __frcp_rn(bs.d);
                bs.enc = isinf(enc) ? kFltMax : enc;
                sfb = bs.sf;
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) x[i] = __fmul_rn(v[i], bs.enc);
                if (SR) {
#pragma unroll
                    for (int hb = 0; hb < 2; ++hb) {
                        const uint4 rb = sr_bits<0u, WIDE>(keys, g + hb);
                        float xs[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) xs[i] = x[8 * hb + i];
                        w[hb] = e2m1x8_sr(xs, rb);
                    }
                } else {
#pragma unroll
                    for (int hb = 0; hb < 2; ++hb)
                        w[hb] = e2m1x8(x[8 * hb], x[8 * hb + 1], x[8 * hb + 2], x[8 * hb + 3], x[8 * hb + 4],
                                       x[8 * hb + 5], x[8 * hb + 6], x[8 * hb + 7]);
                }
            }
            if (valid) *reinterpret_cast<uint2*>(nvp + it * nv_step) = make_uint2(w[0], w[1]);
            sfo_nv[kk][l16] = (uint8_t)sfb;
        }
    }
    __syncthreads();
    // Scale bytes of the tile's output rows: NVFP4 columns m0/16 .. +15, MXFP8
    // columns m0/32 .. +7 of rows k0 .. k0 + 63.  Four consecutive columns
    // form one word of the swizzled layout (its padding absorbs a short last
    // group) or of a row-major row whose length is a multiple of 4; otherwise
    // bytes are stored.
    const int64_t kin = K - k0 < RT_K ? K - k0 : RT_K;
    if (NV) {
        const int kk = tid >> 2, q = tid & 3;
        const int64_t ncols = rows >> 4, col = (m0 >> 4) + 4 * q;
        if (kk < kin && col < ncols) {
            const uint32_t word = *reinterpret_cast<const uint32_t*>(&sfo_nv[kk][4 * q]);
            const int64_t gk = k0 + kk;
            if (SWZ || (ncols & 3) == 0) {
                const int64_t off = SWZ ? sf_swizzled(gk, col, (ncols + 3) >> 2) : gk * ncols + col;
                *reinterpret_cast<uint32_t*>(nv_sf + off) = word;
            } else {
                for (int i = 0; i < 4 && col + i < ncols; ++i) nv_sf[gk * ncols + col + i] = (uint8_t)(word >> (8 * i));
            }
        }
    }
    if (MX && tid < 2 * RT_K) {
        const int kk = tid >> 1, q = tid & 1;
        const int64_t ncols = rows >> 5, col = (m0 >> 5) + 4 * q;
        if (kk < kin && col < ncols) {
            const uint32_t word = *reinterpret_cast<const uint32_t*>(&sfo_mx[kk][4 * q]);
            const int64_t gk = k0 + kk;
            if (SWZ || (ncols & 3) == 0) {
                const int64_t off = SWZ ? sf_swizzled(gk, col, (ncols + 3) >> 2) : gk * ncols + col;
                *reinterpret_cast<uint32_t*>(mx_sf + off) = word;
            } else {
                for (int i = 0; i < 4 && col + i < ncols; ++i) mx_sf[gk * ncols + col + i] = (uint8_t)(word >> (8 * i));
            }
        }
    }
}

template <typename... KArgs, typename... Args>
void launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Both passes; colmax (K words) is cleared first when NVFP4 output is wanted.
cudaError_t requant_passes(const uint8_t* codes, const uint8_t* sf, const float* row_scale, int64_t rows, int64_t K,
                           unsigned int* colmax, uint8_t* nvc, uint8_t* nvs, float* nvt, uint8_t* mxc, uint8_t* mxs,
                           uint64_t seed, bool sr, bool swz, cudaStream_t st)
{
    const bool nv = nvc != nullptr, mx = mxc != nullptr;
    if (nv) {
        cudaError_t err = cudaMemsetAsync(colmax, 0, (size_t)K * sizeof(unsigned int), st);
        if (err != cudaSuccess) return err;
        const int64_t chunks = (K + CM_COLS - 1) / CM_COLS;
        int sms = 148;
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int64_t gy = std::max<int64_t>(1, std::min<int64_t>((4 * (int64_t)sms + chunks - 1) / chunks,
                                                                  (rows / 8 + 7) / 8));
        const dim3 g1((unsigned)chunks, (unsigned)gy);
        if (swz) launch_pdl(k_rq_colmax<true>, g1, dim3(256), st, codes, sf, row_scale, rows, K, colmax);
        else launch_pdl(k_rq_colmax<false>, g1, dim3(256), st, codes, sf, row_scale, rows, K, colmax);
    }
    const dim3 g2((unsigned)((K + RT_K - 1) / RT_K), (unsigned)((rows + RT_M - 1) / RT_M));
    const PhiloxKeys keys = philox_keys(seed);
    const bool wide = (uint64_t)rows * (uint64_t)K > (1ull << 35);  // Philox counters above 2^32
#define BSQ_RQ(S, R, N, M, W)                                                                                    \
    launch_pdl(k_rq_tile<S, R, N, M, W>, g2, dim3(256), st, codes, sf, row_scale, rows, K, colmax, nvc, nvs, nvt, \
               mxc, mxs, keys)
#define BSQ_RQ2(S, R, W)                              \
    do {                                              \
        if (nv && mx) BSQ_RQ(S, R, true, true, W);    \
        else if (nv) BSQ_RQ(S, R, true, false, W);    \
        else BSQ_RQ(S, R, false, true, W);            \
    } while (0)
    if (swz) {
        if (!sr) BSQ_RQ2(true, false, false); else if (wide) BSQ_RQ2(true, true, true); else BSQ_RQ2(true, true, false);
    } else {
        if (!sr) BSQ_RQ2(false, false, false); else if (wide) BSQ_RQ2(false, true, true); else BSQ_RQ2(false, true, false);
    }
#undef BSQ_RQ2
#undef BSQ_RQ
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_requant(const uint8_t* codes, const uint8_t* sf, const float* row_scale, int64_t rows, int64_t K,
                           unsigned int* colmax, uint8_t* nvc, uint8_t* nvs, float* nvt, uint8_t* mxc, uint8_t* mxs,
                           uint64_t seed, bool sr, bool swz, cudaStream_t st)
{
    return requant_passes(codes, sf, row_scale, rows, K, colmax, nvc, nvs, nvt, mxc, mxs, seed, sr, swz, st);
}

// ---------------------------------------------------------------------------
// Allocation-free requantization (requant_transpose_sr_noalloc).
//
// Some callers cannot give the library device memory for scratch: a host
// framework that only owns its input and output buffers, or code that must
// not allocate device memory once it is running.  For them the column maxima
// of |D| live in this file-scope device array instead of a caller workspace.
// Every GPU that loads the library holds it (256 KB) until the process exits,
// every call shares it, and it keeps the last call's contents, so each call
// clears the part it uses first; calls that overlap on the GPU (different
// streams, or different host threads on one device) race on it.
namespace {

constexpr int64_t kNoallocMaxK = 65536;
__device__ __align__(256) unsigned int g_requant_colmax[kNoallocMaxK];

// Device address of g_requant_colmax, looked up once per device with that
// device current (the host-side name is only a stand-in for it).
constexpr int kNoallocDevices = 64;
std::mutex g_noalloc_mutex;
unsigned int* g_noalloc_ptr[kNoallocDevices];

cudaError_t noalloc_scratch(unsigned int** out)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kNoallocDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_requant_colmax);
        if (err != cudaSuccess) return err;
        g_noalloc_ptr[dev] = static_cast<unsigned int*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace

int64_t noalloc_requant_max_k() { return kNoallocMaxK; }

cudaError_t launch_requant_noalloc(const uint8_t* codes, const uint8_t* sf, const float* row_scale, int64_t rows,
                                   int64_t K, uint8_t* nvc, uint8_t* nvs, float* nvt, uint8_t* mxc, uint8_t* mxs,
                                   uint64_t seed, bool sr, bool swz, cudaStream_t st)
{
    unsigned int* colmax = nullptr;
    cudaError_t err = noalloc_scratch(&colmax);
    if (err != cudaSuccess) return err;
    return requant_passes(codes, sf, row_scale, rows, K, colmax, nvc, nvs, nvt, mxc, mxs, seed, sr, swz, st);
}

}  // namespace bsq
