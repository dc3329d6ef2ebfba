// quant.cu -- bandwidth-bound quantizers: per-token / per-expert NVFP4,
// MXFP8 row+column copies, dequantize-transpose-requantize with Philox
// stochastic rounding, and small helper kernels (SF layout conversion,
// format probes, random-bit dumps).
//
// Design for GB300: every kernel streams its input once with 16-byte
// coalesced loads (ld.global.nc, no L1 allocation), reduces maxima with
// integer operations on bf16 magnitude bits and warp shuffles, and writes
// packed codes with 8- to 32-byte stores.  Grids are sized in multiples of
// the SM count.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace bsq {

BSQ_DEVICE uint4 ldg_stream(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

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

// One 16-element block -> codes (2 words) and SF byte, per-row scale t.
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

BSQ_DEVICE void store_sf(uint8_t* sf, bool swz, int64_t row, int64_t col, int64_t ncols, uint32_t v)
{
    const int64_t off = swz ? sf_swizzled(row, col, (ncols + 3) >> 2) : row * ncols + col;
    sf[off] = (uint8_t)v;
}

// ---------------------------------------------------------------------------
// Per-row NVFP4, one warp per row.  Lane l owns blocks l, l+32, ... (BPL of
// them); the warp reads 1 KB contiguous per step.  TMODE 0: per-row scale from
// the row maximum; TMODE 1: per-group scale from group_amax[row / rpg].
// With SWZ the padding rows up to a multiple of 128 and the padding SF
// columns are written as 0.
template <int BPL, bool FOUR_SIX, bool SWZ, int TMODE>
__global__ void __launch_bounds__(256) k_nvfp4_rows(const uint16_t* __restrict__ x, int64_t rows, int64_t K,
                                                    int64_t ldx, uint8_t* __restrict__ codes,
                                                    uint8_t* __restrict__ sf, float* __restrict__ row_scale,
                                                    const float* __restrict__ group_amax, int64_t rpg)
{
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nblk = (int)(K >> 4);
    const int ncol_pad = SWZ ? ((nblk + 3) & ~3) : nblk;
    const int64_t rows_iter = SWZ ? ((rows + 127) & ~(int64_t)127) : rows;
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows_iter; r += nwarps) {
        if (r >= rows) {  // swizzle padding rows
            for (int b = lane; b < ncol_pad; b += 32) store_sf(sf, SWZ, r, b, nblk, 0u);
            continue;
        }
        const uint16_t* xr = x + r * ldx;
        uint4 va[BPL], vb[BPL];
        uint32_t bmax[BPL];
        uint32_t rmax = 0;
#pragma unroll
        for (int i = 0; i < BPL; ++i) {
            const int b = lane + 32 * i;
            if (b < nblk) {
                va[i] = ldg_stream(xr + 16 * b);
                vb[i] = ldg_stream(xr + 16 * b + 8);
            } else {
                va[i] = vb[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int i = 0; i < BPL; ++i) {
            bmax[i] = absmax16(va[i], vb[i]);
            rmax = max(rmax, bmax[i]);
        }
        float t;
        if (TMODE == 0) {
            rmax = __reduce_max_sync(0xFFFFFFFFu, rmax);
            t = __fdiv_rn(bf16mag_to_f32(rmax), kNvfp4ScaleDivisor);
            if (lane == 0) row_scale[r] = t;
        } else {
            t = __fdiv_rn(group_amax[r / rpg], kNvfp4ScaleDivisor);
        }
        const float six_t = __fmul_rn(6.0f, t), four_t = __fmul_rn(4.0f, t);
        uint2* crow = reinterpret_cast<uint2*>(codes + r * (K >> 1));
#pragma unroll
        for (int i = 0; i < BPL; ++i) {
            const int b = lane + 32 * i;
            if (b < nblk) {
                uint2 c;
                uint32_t s;
                nvfp4_block<FOUR_SIX>(va[i], vb[i], bmax[i], t, six_t, four_t, c, s);
                crow[b] = c;
                store_sf(sf, SWZ, r, b, nblk, s);
            } else if (SWZ && b < ncol_pad) {
                store_sf(sf, SWZ, r, b, nblk, 0u);
            }
        }
    }
}

// Long rows (K > 8192): two passes over the row, chunk by chunk.
template <bool FOUR_SIX, bool SWZ, int TMODE>
__global__ void __launch_bounds__(256) k_nvfp4_rows_long(const uint16_t* __restrict__ x, int64_t rows, int64_t K,
                                                         int64_t ldx, uint8_t* __restrict__ codes,
                                                         uint8_t* __restrict__ sf, float* __restrict__ row_scale,
                                                         const float* __restrict__ group_amax, int64_t rpg)
{
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nblk = (int)(K >> 4);
    const int ncol_pad = SWZ ? ((nblk + 3) & ~3) : nblk;
    const int64_t rows_iter = SWZ ? ((rows + 127) & ~(int64_t)127) : rows;
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows_iter; r += nwarps) {
        if (r >= rows) {
            for (int b = lane; b < ncol_pad; b += 32) store_sf(sf, SWZ, r, b, nblk, 0u);
            continue;
        }
        const uint16_t* xr = x + r * ldx;
        float t;
        if (TMODE == 0) {
            uint32_t rmax = 0;
            for (int b = lane; b < nblk; b += 32) rmax = max(rmax, absmax16(ldg_stream(xr + 16 * b), ldg_stream(xr + 16 * b + 8)));
            rmax = __reduce_max_sync(0xFFFFFFFFu, rmax);
            t = __fdiv_rn(bf16mag_to_f32(rmax), kNvfp4ScaleDivisor);
            if (lane == 0) row_scale[r] = t;
        } else {
            t = __fdiv_rn(group_amax[r / rpg], kNvfp4ScaleDivisor);
        }
        const float six_t = __fmul_rn(6.0f, t), four_t = __fmul_rn(4.0f, t);
        uint2* crow = reinterpret_cast<uint2*>(codes + r * (K >> 1));
        for (int b = lane; b < ncol_pad; b += 32) {
            if (b < nblk) {
                const uint4 a = ldg_stream(xr + 16 * b), c2 = ldg_stream(xr + 16 * b + 8);
                uint2 c;
                uint32_t s;
                nvfp4_block<FOUR_SIX>(a, c2, absmax16(a, c2), t, six_t, four_t, c, s);
                crow[b] = c;
                store_sf(sf, SWZ, r, b, nblk, s);
            } else {
                store_sf(sf, SWZ, r, b, nblk, 0u);
            }
        }
    }
}

// Per-group maximum |x| (bits of a non-negative float, so an unsigned
// atomicMax orders them) into group_amax (zeroed by the caller).
__global__ void __launch_bounds__(256) k_group_amax(const uint16_t* __restrict__ x, int64_t rows, int64_t K,
                                                    int64_t rpg, unsigned int* __restrict__ group_amax)
{
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nblk = (int)(K >> 4);
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += nwarps) {
        const uint16_t* xr = x + r * K;
        uint32_t m = 0;
        for (int b = lane; b < nblk; b += 32) m = max(m, absmax16(ldg_stream(xr + 16 * b), ldg_stream(xr + 16 * b + 8)));
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0 && m) atomicMax(group_amax + r / rpg, m << 16);
    }
}

__global__ void k_group_finalize(float* __restrict__ scale, int64_t groups)
{
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g < groups) scale[g] = __fdiv_rn(scale[g], kNvfp4ScaleDivisor);
}

// ---------------------------------------------------------------------------
// MXFP8 row + column copies.  CTA tile 128 rows x 128 columns, 512 threads.
// Row copy straight from registers (4 lanes per 32-element block); the tile is
// staged in shared memory (rows padded by 16 bytes) for the column copy, where
// a warp reads 32 adjacent columns of one row per step.
constexpr int MX_TILE = 128;
constexpr int MX_LD = MX_TILE + 8;  // bf16 elements per staged row

template <bool SWZ, bool ROW, bool COL>
__global__ void __launch_bounds__(512) k_mxfp8_rowcol(const uint16_t* __restrict__ x, int64_t rows, int64_t K,
                                                      int64_t ldx, uint8_t* __restrict__ row_codes,
                                                      uint8_t* __restrict__ row_sf, uint8_t* __restrict__ col_codes,
                                                      uint8_t* __restrict__ col_sf)
{
    __shared__ __align__(16) uint16_t tile[MX_TILE * MX_LD];
    const int tid = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.y * MX_TILE, col0 = (int64_t)blockIdx.x * MX_TILE;
    const int64_t nsf_row = K >> 5, nsf_col = rows >> 5;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int item = tid + 512 * i;
        const int r = item >> 4, ch = item & 15;
        const int64_t gr = row0 + r, gc = col0 + 8 * ch;
        const bool ok = gr < rows && gc < K;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (ok) v = ldg_stream(x + gr * ldx + gc);
        if (COL) *reinterpret_cast<uint4*>(tile + r * MX_LD + 8 * ch) = v;
        if (ROW) {
            uint32_t m = absmax_bf16x2(0u, v.x);
            m = absmax_bf16x2(m, v.y);
            m = absmax_bf16x2(m, v.z);
            m = absmax_bf16x2(m, v.w);
            m = fold_halves(m);
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            if (ok) {
                uint2 c = make_uint2(0u, 0u);
                uint32_t s = 0;
                if (m) {
                    const int X = mx_exponent(m << 16);
                    const float mul = mx_multiplier(X);
                    s = (uint32_t)(X + 127);
                    c.x = e4m3x4(__fmul_rn(bf16_lo(v.x), mul), __fmul_rn(bf16_hi(v.x), mul),
                                 __fmul_rn(bf16_lo(v.y), mul), __fmul_rn(bf16_hi(v.y), mul));
                    c.y = e4m3x4(__fmul_rn(bf16_lo(v.z), mul), __fmul_rn(bf16_hi(v.z), mul),
                                 __fmul_rn(bf16_lo(v.w), mul), __fmul_rn(bf16_hi(v.w), mul));
                }
                *reinterpret_cast<uint2*>(row_codes + gr * K + gc) = c;
                if ((ch & 3) == 0) store_sf(row_sf, SWZ, gr, gc >> 5, nsf_row, s);
            }
        }
    }
    if (!COL) return;
    __syncthreads();
    const int c = tid & 127, rb = tid >> 7;
    const int64_t gc = col0 + c, gr = row0 + 32 * rb;
    if (gc >= K || gr >= rows) return;
    float v[32];
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t b = tile[(32 * rb + i) * MX_LD + c];
        m = max(m, b & 0x7FFFu);
        v[i] = __uint_as_float(b << 16);
    }
    uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = o0;
    uint32_t s = 0;
    if (m) {
        const int X = mx_exponent(m << 16);
        const float mul = mx_multiplier(X);
        s = (uint32_t)(X + 127);
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            w[j] = e4m3x4(__fmul_rn(v[4 * j], mul), __fmul_rn(v[4 * j + 1], mul), __fmul_rn(v[4 * j + 2], mul),
                          __fmul_rn(v[4 * j + 3], mul));
        o0 = make_uint4(w[0], w[1], w[2], w[3]);
        o1 = make_uint4(w[4], w[5], w[6], w[7]);
    }
    uint4* dst = reinterpret_cast<uint4*>(col_codes + gc * rows + gr);
    dst[0] = o0;
    dst[1] = o1;
    store_sf(col_sf, SWZ, gc, gr >> 5, nsf_col, s);
}

// Zero the padding of a swizzled SF buffer (rows and columns beyond the
// data up to the tile boundaries).
__global__ void k_sf_pad_zero(uint8_t* __restrict__ sf, int64_t rows, int64_t cols)
{
    const int64_t rpad = (rows + 127) & ~(int64_t)127, cpad = (cols + 3) & ~(int64_t)3;
    const int64_t n = rpad * cpad;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / cpad, c = i % cpad;
        if (r >= rows || c >= cols) sf[sf_swizzled(r, c, cpad >> 2)] = 0;
    }
}

// ---------------------------------------------------------------------------
// Requant pass 1: per-column maximum of |D|, D = rn(rn(e2m1 * sf) * t), in
// two deterministic stages.  Stage A: a thread owns 8 columns (one code word)
// of a chunk of RQ_CHUNK rows and writes the chunk maxima to
// part[chunk][K].  Stage B: one thread per column reduces over the chunks.
constexpr int RQ_CHUNK = 32;
constexpr int RQ_COLMAX_THREADS = 128;

template <bool SWZ>
__global__ void __launch_bounds__(RQ_COLMAX_THREADS) k_requant_colmax_part(const uint8_t* __restrict__ codes,
                                                                           const uint8_t* __restrict__ sf,
                                                                           const float* __restrict__ row_scale,
                                                                           int64_t rows, int64_t K,
                                                                           float* __restrict__ part)
{
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // column group of 8
    if (g >= (K >> 3)) return;
    const int64_t r0 = (int64_t)blockIdx.y * RQ_CHUNK;
    const int64_t nsf = K >> 4;
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = 0.0f;
    const uint32_t* cw = reinterpret_cast<const uint32_t*>(codes);
#pragma unroll 8
    for (int j = 0; j < RQ_CHUNK; ++j) {
        const int64_t r = r0 + j;
        if (r >= rows) break;
        const uint32_t w = __ldg(cw + r * (K >> 3) + g);
        const int64_t so = SWZ ? sf_swizzled(r, g >> 1, (nsf + 3) >> 2) : r * nsf + (g >> 1);
        const float s = e4m3_to_f32(__ldg(sf + so));
        const float t = __ldg(row_scale + r);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float a = e2m1_to_f32((w >> (4 * i)) & 7u);
            m[i] = fmaxf(m[i], __fmul_rn(__fmul_rn(a, s), t));
        }
    }
    float4* dst = reinterpret_cast<float4*>(part + (int64_t)blockIdx.y * K + 8 * g);
    dst[0] = make_float4(m[0], m[1], m[2], m[3]);
    dst[1] = make_float4(m[4], m[5], m[6], m[7]);
}

__global__ void __launch_bounds__(256) k_requant_colmax_reduce(const float* __restrict__ part, int64_t nchunks,
                                                               int64_t K, unsigned int* __restrict__ colmax)
{
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= K) return;
    float m = 0.0f;
    for (int64_t j = 0; j < nchunks; ++j) m = fmaxf(m, __ldg(part + j * K + c));
    colmax[c] = __float_as_uint(m);
}

// Requant pass 2.  CTA tile: 128 source rows (m) x 64 source columns (k),
// 256 threads.  The tile is dequantized into shared memory (binary32), then
// each thread produces one 32-element run of one output row (a source
// column): the MXFP8 block and two NVFP4 blocks, with RNE or Philox SR.
constexpr int RQ_TM = 128, RQ_TK = 64;

template <bool SWZ, bool SR, bool NV, bool MX>
__global__ void __launch_bounds__(256) k_requant_main(const uint8_t* __restrict__ codes,
                                                      const uint8_t* __restrict__ sf,
                                                      const float* __restrict__ row_scale, int64_t rows, int64_t K,
                                                      const unsigned int* __restrict__ colmax,
                                                      uint8_t* __restrict__ nv_codes, uint8_t* __restrict__ nv_sf,
                                                      float* __restrict__ nv_scale, uint8_t* __restrict__ mx_codes,
                                                      uint8_t* __restrict__ mx_sf, uint64_t seed)
{
    __shared__ __align__(16) float D[RQ_TM * RQ_TK];
    const int tid = threadIdx.x;
    const int64_t m0 = (int64_t)blockIdx.y * RQ_TM, k0 = (int64_t)blockIdx.x * RQ_TK;
    const int64_t nsf_in = K >> 4;
    const uint32_t* cw = reinterpret_cast<const uint32_t*>(codes);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int item = tid + 256 * i;
        const int m = item >> 3, g = item & 7;
        const int64_t gm = m0 + m, gk = k0 + 8 * g;
        float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
        if (gm < rows && gk < K) {
            const uint32_t w = __ldg(cw + gm * (K >> 3) + (gk >> 3));
            const int64_t so = SWZ ? sf_swizzled(gm, gk >> 4, (nsf_in + 3) >> 2) : gm * nsf_in + (gk >> 4);
            const float s = e4m3_to_f32(__ldg(sf + so));
            const float t = __ldg(row_scale + gm);
            float d[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) d[j] = __fmul_rn(__fmul_rn(e2m1_to_f32((w >> (4 * j)) & 0xFu), s), t);
            lo = make_float4(d[0], d[1], d[2], d[3]);
            hi = make_float4(d[4], d[5], d[6], d[7]);
        }
        float4* dst = reinterpret_cast<float4*>(D + m * RQ_TK + 8 * g);
        dst[0] = lo;
        dst[1] = hi;
    }
    __syncthreads();
    const int c = tid & 63, mb = tid >> 6;
    const int64_t gk = k0 + c, gm = m0 + 32 * mb;
    if (gk >= K || gm >= rows) return;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = D[(32 * mb + i) * RQ_TK + c];
    const uint64_t idx0 = (uint64_t)gk * (uint64_t)rows + (uint64_t)gm;  // index in Y of v[0]
    if (MX) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
        uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        uint32_t s = 0;
        if (amax > 0.f) {
            const int X = mx_exponent(__float_as_uint(amax));
            const float mul = mx_multiplier(X);
            s = (uint32_t)(X + 127);
            if (SR) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 rb = sr_block_bits(seed, 1u, (idx0 >> 3) + q);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t code = e4m3_sr(__fmul_rn(v[8 * q + j], mul), sr_pick16(rb, j));
                        w[2 * q + (j >> 2)] |= code << (8 * (j & 3));
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    w[j] = e4m3x4(__fmul_rn(v[4 * j], mul), __fmul_rn(v[4 * j + 1], mul),
                                  __fmul_rn(v[4 * j + 2], mul), __fmul_rn(v[4 * j + 3], mul));
            }
        }
        uint4* dst = reinterpret_cast<uint4*>(mx_codes + gk * rows + gm);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        store_sf(mx_sf, SWZ, gk, gm >> 5, rows >> 5, s);
    }
    if (NV) {
        const float t = __fdiv_rn(__uint_as_float(__ldg(colmax + gk)), kNvfp4ScaleDivisor);
        if (blockIdx.y == 0 && mb == 0) nv_scale[gk] = t;
        const float six_t = __fmul_rn(6.0f, t);
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        uint32_t sfb[2] = {0u, 0u};
        if (t != 0.0f) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float* xb = v + 16 * h;
                float ab = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(xb[i]));
                const BlockScale bs = nvfp4_block_scale(ab, six_t, t);
                sfb[h] = bs.sf;
                if (SR) {
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const uint4 rb = sr_block_bits(seed, 0u, (idx0 >> 3) + 2 * h + q);
                        uint32_t word = 0;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            word |= e2m1_sr(__fmul_rn(xb[8 * q + j], bs.enc), sr_pick16(rb, j)) << (4 * j);
                        w[2 * h + q] = word;
                    }
                } else {
                    const uint2 cc = encode16(xb, bs.enc);
                    w[2 * h] = cc.x;
                    w[2 * h + 1] = cc.y;
                }
            }
        }
        *reinterpret_cast<uint4*>(nv_codes + gk * (rows >> 1) + (gm >> 1)) = make_uint4(w[0], w[1], w[2], w[3]);
        store_sf(nv_sf, SWZ, gk, gm >> 4, rows >> 4, sfb[0]);
        store_sf(nv_sf, SWZ, gk, (gm >> 4) + 1, rows >> 4, sfb[1]);
    }
}

// ---------------------------------------------------------------------------
// Helpers.
__global__ void k_sf_swizzle(const uint8_t* __restrict__ in, int64_t rows, int64_t cols, uint8_t* __restrict__ out,
                             int dir)
{
    const int64_t rpad = (rows + 127) & ~(int64_t)127, cpad = (cols + 3) & ~(int64_t)3;
    const int64_t n = rpad * cpad;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / cpad, c = i % cpad;
        const int64_t so = sf_swizzled(r, c, cpad >> 2);
        const bool data = r < rows && c < cols;
        if (dir == 0)
            out[so] = data ? in[r * cols + c] : 0;
        else if (data)
            out[r * cols + c] = in[so];
    }
}

__global__ void k_format_probe(int kind, const float* __restrict__ in, const uint32_t* __restrict__ rbits,
                               void* __restrict__ out, int64_t n)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float v = in[i];
        switch (kind) {
            case 0: static_cast<uint8_t*>(out)[i] = (uint8_t)(e2m1x8(v, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f) & 0xFu); break;
            case 1: static_cast<uint8_t*>(out)[i] = (uint8_t)e4m3_rn(v); break;
            case 2: static_cast<uint8_t*>(out)[i] = (uint8_t)e2m1_sr(v, rbits[i] & 0xFFFFu); break;
            case 3: static_cast<uint8_t*>(out)[i] = (uint8_t)e4m3_sr(v, rbits[i] & 0xFFFFu); break;
            case 4: static_cast<float*>(out)[i] = e2m1_to_f32(__float_as_uint(v) & 0xFu); break;
            default: static_cast<float*>(out)[i] = e4m3_to_f32(__float_as_uint(v) & 0xFFu); break;
        }
    }
}

__global__ void k_philox_bits16(uint64_t seed, uint32_t stream, uint64_t idx0, int64_t n, uint16_t* __restrict__ out)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t idx = idx0 + (uint64_t)i;
        const uint4 w = sr_block_bits(seed, stream, idx >> 3);
        out[i] = (uint16_t)sr_pick16(w, (int)(idx & 7));
    }
}

// ---------------------------------------------------------------------------
// Launchers.
static int grid_for(int64_t warps_needed, int sms)
{
    const int64_t blocks = (warps_needed + 7) / 8;
    const int64_t cap = (int64_t)sms * 16;
    return (int)std::max<int64_t>(1, std::min<int64_t>(blocks, cap));
}

template <bool F46, bool SWZ, int TM>
static void launch_rows_t(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx, uint8_t* codes, uint8_t* sf,
                          float* rs, const float* gam, int64_t rpg, int sms, cudaStream_t st)
{
    const int nblk = (int)(K >> 4);
    const int64_t rows_iter = SWZ ? ((rows + 127) & ~(int64_t)127) : rows;
    const int grid = grid_for(rows_iter, sms);
    if (nblk <= 32)
        k_nvfp4_rows<1, F46, SWZ, TM><<<grid, 256, 0, st>>>(x, rows, K, ldx, codes, sf, rs, gam, rpg);
    else if (nblk <= 64)
        k_nvfp4_rows<2, F46, SWZ, TM><<<grid, 256, 0, st>>>(x, rows, K, ldx, codes, sf, rs, gam, rpg);
    else if (nblk <= 128)
        k_nvfp4_rows<4, F46, SWZ, TM><<<grid, 256, 0, st>>>(x, rows, K, ldx, codes, sf, rs, gam, rpg);
    else if (nblk <= 256)
        k_nvfp4_rows<8, F46, SWZ, TM><<<grid, 256, 0, st>>>(x, rows, K, ldx, codes, sf, rs, gam, rpg);
    else if (nblk <= 512)
        k_nvfp4_rows<16, F46, SWZ, TM><<<grid, 256, 0, st>>>(x, rows, K, ldx, codes, sf, rs, gam, rpg);
    else
        k_nvfp4_rows_long<F46, SWZ, TM><<<grid, 256, 0, st>>>(x, rows, K, ldx, codes, sf, rs, gam, rpg);
}

void launch_nvfp4_rows(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx, uint8_t* codes, uint8_t* sf,
                       float* row_scale, const float* group_amax, int64_t rpg, bool four_six, bool swz, int sms,
                       cudaStream_t st)
{
    const bool per_group = group_amax != nullptr;
#define BSQ_ROWS(F, S, T) launch_rows_t<F, S, T>(x, rows, K, ldx, codes, sf, row_scale, group_amax, rpg, sms, st)
    if (per_group) {
        if (swz) BSQ_ROWS(false, true, 1); else BSQ_ROWS(false, false, 1);
    } else if (four_six) {
        if (swz) BSQ_ROWS(true, true, 0); else BSQ_ROWS(true, false, 0);
    } else {
        if (swz) BSQ_ROWS(false, true, 0); else BSQ_ROWS(false, false, 0);
    }
#undef BSQ_ROWS
}

void launch_group_amax(const uint16_t* x, int64_t rows, int64_t K, int64_t rpg, float* group_amax, int sms,
                       cudaStream_t st)
{
    k_group_amax<<<grid_for(rows, sms), 256, 0, st>>>(x, rows, K, rpg, reinterpret_cast<unsigned int*>(group_amax));
}

void launch_group_finalize(float* scale, int64_t groups, cudaStream_t st)
{
    k_group_finalize<<<(int)((groups + 255) / 256), 256, 0, st>>>(scale, groups);
}

void launch_mxfp8_rowcol(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx, uint8_t* rc, uint8_t* rs,
                         uint8_t* cc, uint8_t* cs, bool swz, cudaStream_t st)
{
    dim3 grid((unsigned)((K + MX_TILE - 1) / MX_TILE), (unsigned)((rows + MX_TILE - 1) / MX_TILE));
    const bool row = rc != nullptr, col = cc != nullptr;
#define BSQ_MX(S, R, C) k_mxfp8_rowcol<S, R, C><<<grid, 512, 0, st>>>(x, rows, K, ldx, rc, rs, cc, cs)
    if (swz) {
        if (row && col) BSQ_MX(true, true, true); else if (row) BSQ_MX(true, true, false); else BSQ_MX(true, false, true);
    } else {
        if (row && col) BSQ_MX(false, true, true); else if (row) BSQ_MX(false, true, false); else BSQ_MX(false, false, true);
    }
#undef BSQ_MX
}

void launch_sf_pad_zero(uint8_t* sf, int64_t rows, int64_t cols, int sms, cudaStream_t st)
{
    if ((rows & 127) == 0 && (cols & 3) == 0) return;
    k_sf_pad_zero<<<sms * 4, 256, 0, st>>>(sf, rows, cols);
}

void launch_requant(const uint8_t* codes, const uint8_t* sf, const float* row_scale, int64_t rows, int64_t K,
                    unsigned int* colmax, uint8_t* nvc, uint8_t* nvs, float* nvt, uint8_t* mxc, uint8_t* mxs,
                    uint64_t seed, bool sr, bool swz, cudaStream_t st)
{
    const bool nv = nvc != nullptr, mx = mxc != nullptr;
    if (nv) {
        // workspace: colmax [K] then the per-chunk maxima [nchunks][K]
        const int64_t nchunks = (rows + RQ_CHUNK - 1) / RQ_CHUNK;
        float* part = reinterpret_cast<float*>(colmax) + ((K + 63) & ~(int64_t)63);
        dim3 g1((unsigned)(((K >> 3) + RQ_COLMAX_THREADS - 1) / RQ_COLMAX_THREADS), (unsigned)nchunks);
        if (swz) k_requant_colmax_part<true><<<g1, RQ_COLMAX_THREADS, 0, st>>>(codes, sf, row_scale, rows, K, part);
        else k_requant_colmax_part<false><<<g1, RQ_COLMAX_THREADS, 0, st>>>(codes, sf, row_scale, rows, K, part);
        k_requant_colmax_reduce<<<(unsigned)((K + 255) / 256), 256, 0, st>>>(part, nchunks, K, colmax);
    }
    dim3 g2((unsigned)((K + RQ_TK - 1) / RQ_TK), (unsigned)((rows + RQ_TM - 1) / RQ_TM));
#define BSQ_RQ(S, R, N, M)                                                                                   \
    k_requant_main<S, R, N, M><<<g2, 256, 0, st>>>(codes, sf, row_scale, rows, K, colmax, nvc, nvs, nvt, mxc, mxs, \
                                                   seed)
#define BSQ_RQ2(S, R)                          \
    do {                                       \
        if (nv && mx) BSQ_RQ(S, R, true, true); \
        else if (nv) BSQ_RQ(S, R, true, false); \
        else BSQ_RQ(S, R, false, true);        \
    } while (0)
    if (swz) {
        if (sr) BSQ_RQ2(true, true); else BSQ_RQ2(true, false);
    } else {
        if (sr) BSQ_RQ2(false, true); else BSQ_RQ2(false, false);
    }
#undef BSQ_RQ2
#undef BSQ_RQ
}

void launch_sf_swizzle(const uint8_t* in, int64_t rows, int64_t cols, uint8_t* out, int dir, int sms,
                       cudaStream_t st)
{
    k_sf_swizzle<<<sms * 4, 256, 0, st>>>(in, rows, cols, out, dir);
}

void launch_format_probe(int kind, const float* in, const uint32_t* rbits, void* out, int64_t n, int sms,
                         cudaStream_t st)
{
    k_format_probe<<<sms * 8, 256, 0, st>>>(kind, in, rbits, out, n);
}

void launch_philox_bits16(uint64_t seed, uint32_t stream, uint64_t idx0, int64_t n, uint16_t* out, int sms,
                          cudaStream_t st)
{
    k_philox_bits16<<<sms * 8, 256, 0, st>>>(seed, stream, idx0, n, out);
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
constexpr int kNoallocRows = 64;  // rows per CTA of the column-maximum pass
__device__ __align__(256) unsigned int g_requant_colmax[kNoallocMaxK];

// Column maxima of |D| straight into the shared array: a thread owns 8
// columns of kNoallocRows rows and folds them in with unsigned atomicMax on
// the bits of non-negative floats (order-independent, so deterministic).
template <bool SWZ>
__global__ void __launch_bounds__(128) k_requant_colmax_atomic(const uint8_t* __restrict__ codes,
                                                               const uint8_t* __restrict__ sf,
                                                               const float* __restrict__ row_scale, int64_t rows,
                                                               int64_t K, unsigned int* __restrict__ colmax)
{
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= (K >> 3)) return;
    const int64_t r0 = (int64_t)blockIdx.y * kNoallocRows;
    const int64_t nsf = K >> 4;
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = 0.0f;
    const uint32_t* cw = reinterpret_cast<const uint32_t*>(codes);
#pragma unroll 8
    for (int j = 0; j < kNoallocRows; ++j) {
        const int64_t r = r0 + j;
        if (r >= rows) break;
        const uint32_t w = __ldg(cw + r * (K >> 3) + g);
        const int64_t so = SWZ ? sf_swizzled(r, g >> 1, (nsf + 3) >> 2) : r * nsf + (g >> 1);
        const float s = e4m3_to_f32(__ldg(sf + so));
        const float t = __ldg(row_scale + r);
#pragma unroll
        for (int i = 0; i < 8; ++i) m[i] = fmaxf(m[i], __fmul_rn(__fmul_rn(e2m1_to_f32((w >> (4 * i)) & 7u), s), t));
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (m[i] > 0.0f) atomicMax(colmax + 8 * g + i, __float_as_uint(m[i]));
}

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
    const bool nv = nvc != nullptr, mx = mxc != nullptr;
    if (nv) {
        err = cudaMemsetAsync(colmax, 0, (size_t)K * sizeof(unsigned int), st);
        if (err != cudaSuccess) return err;
        dim3 g1((unsigned)(((K >> 3) + 127) / 128), (unsigned)((rows + kNoallocRows - 1) / kNoallocRows));
        if (swz) k_requant_colmax_atomic<true><<<g1, 128, 0, st>>>(codes, sf, row_scale, rows, K, colmax);
        else k_requant_colmax_atomic<false><<<g1, 128, 0, st>>>(codes, sf, row_scale, rows, K, colmax);
    }
    dim3 g2((unsigned)((K + RQ_TK - 1) / RQ_TK), (unsigned)((rows + RQ_TM - 1) / RQ_TM));
#define BSQ_RQN(S, R, N, M)                                                                                   \
    k_requant_main<S, R, N, M><<<g2, 256, 0, st>>>(codes, sf, row_scale, rows, K, colmax, nvc, nvs, nvt, mxc, mxs, \
                                                   seed)
#define BSQ_RQN2(S, R)                            \
    do {                                          \
        if (nv && mx) BSQ_RQN(S, R, true, true);  \
        else if (nv) BSQ_RQN(S, R, true, false);  \
        else BSQ_RQN(S, R, false, true);          \
    } while (0)
    if (swz) {
        if (sr) BSQ_RQN2(true, true); else BSQ_RQN2(true, false);
    } else {
        if (sr) BSQ_RQN2(false, true); else BSQ_RQN2(false, false);
    }
#undef BSQ_RQN2
#undef BSQ_RQN
    return cudaGetLastError();
}

}  // namespace bsq
