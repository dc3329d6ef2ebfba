// quant.cu -- bandwidth-bound quantizers: per-token / per-expert NVFP4,
// MXFP8 row+column copies, the Hadamard-transform and 2-D quantizers, the
// dequantizer, and small helper kernels (SF layout conversion, format
// probes, random-bit dumps).  The backward requantization is in requant.cu.
//
// Design for GB300: every kernel streams its input once with 16-byte
// coalesced loads (ld.global.nc, no L1 allocation), reduces maxima with
// integer operations on bf16 magnitude bits and warp shuffles, and writes
// packed codes with 8- to 32-byte stores.  Grids are sized in multiples of
// the SM count.

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

BSQ_DEVICE void store_sf(uint8_t* sf, bool swz, int64_t row, int64_t col, int64_t ncols, uint32_t v)
{
    const int64_t off = swz ? sf_swizzled(row, col, (ncols + 3) >> 2) : row * ncols + col;
    sf[off] = (uint8_t)v;
}

// ---------------------------------------------------------------------------
// Per-row NVFP4 with LPR lanes per row (32: one warp per row; 16: each
// half-warp takes a row, for row lengths whose block count is an odd multiple
// of 16, so no lane idles).  Lane l of a row owns blocks l, l+LPR, ... (BPL of
// them) and reads them with 16-byte streaming loads.  TMODE 0: per-row scale
// from the row maximum; TMODE 1: per-group scale from group_amax[row / rpg].
// With SWZ the padding rows up to a multiple of 128 and the padding SF
// columns are written as 0.  The 4/6 form with swizzled scale factors and
// four blocks a lane is held to 80 registers (3 CTAs of 256 threads an SM;
// left free it takes 105 and an SM holds 16 warps instead of 24).
template <int BPL, bool FOUR_SIX, bool SWZ, int TMODE, int LPR = 32>
__global__ void __launch_bounds__(256, (FOUR_SIX && SWZ && BPL == 4) ? 3 : 0) k_nvfp4_rows(const uint16_t* __restrict__ x, int64_t rows, int64_t K,
                                                    int64_t ldx, uint8_t* __restrict__ codes,
                                                    uint8_t* __restrict__ sf, float* __restrict__ row_scale,
                                                    const float* __restrict__ group_amax, int64_t rpg)
{
    pdl_enter();
    constexpr int RPW = 32 / LPR;  // rows per warp step
    const int lane = threadIdx.x & 31, lr = lane % LPR;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nblk = (int)(K >> 4);
    const int ncol_pad = SWZ ? ((nblk + 3) & ~3) : nblk;
    const int64_t rows_iter = SWZ ? ((rows + 127) & ~(int64_t)127) : rows;
    // warp-uniform loop over groups of RPW rows (the shuffles below need all lanes)
    for (int64_t r0 = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * RPW; r0 < rows_iter;
         r0 += nwarps * RPW) {
        const int64_t r = r0 + lane / LPR;
        const bool in_iter = r < rows_iter, real = r < rows;
        if (in_iter && !real) {  // swizzle padding rows
            for (int b = lr; b < ncol_pad; b += LPR) store_sf(sf, SWZ, r, b, nblk, 0u);
        }
        const uint16_t* xr = x + r * ldx;
        uint4 va[BPL], vb[BPL];
        uint32_t bmax[BPL];
        uint32_t rmax = 0;
#pragma unroll
        for (int i = 0; i < BPL; ++i) {
            const int b = lr + LPR * i;
            if (real && b < nblk) {
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
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) rmax = max(rmax, __shfl_xor_sync(0xFFFFFFFFu, rmax, off));
            t = __fdiv_rn(bf16mag_to_f32(rmax), kNvfp4ScaleDivisor);
            if (lr == 0 && real) row_scale[r] = t;
        } else {
            t = real ? __fdiv_rn(group_amax[r / rpg], kNvfp4ScaleDivisor) : 0.0f;
        }
        if (!real) continue;
        const float six_t = __fmul_rn(6.0f, t), four_t = __fmul_rn(4.0f, t);
        uint2* crow = reinterpret_cast<uint2*>(codes + r * (K >> 1));
#pragma unroll
        for (int i = 0; i < BPL; ++i) {
            const int b = lr + LPR * i;
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

// Wide rows (128 < blocks <= 512): four warps per row, up to four blocks per
// lane (one warp per row would need 8-16 blocks per lane, i.e. more registers
// and so fewer warps in flight).  A CTA of 8 warps takes 2 rows per step; the
// row maximum is folded across the row's warps in shared memory.  Lane l of
// part p owns blocks 32 p + l + 128 i.  The 4/6 form with swizzled scale
// factors is held to 80 registers, as in k_nvfp4_rows.
template <bool FOUR_SIX, bool SWZ, int TMODE>
__global__ void __launch_bounds__(256, (FOUR_SIX && SWZ) ? 3 : 0) k_nvfp4_rows_wide(const uint16_t* __restrict__ x, int64_t rows, int64_t K,
                                                         int64_t ldx, uint8_t* __restrict__ codes,
                                                         uint8_t* __restrict__ sf, float* __restrict__ row_scale,
                                                         const float* __restrict__ group_amax, int64_t rpg)
{
    pdl_enter();
    constexpr int WPR = 4, BPL = 4;
    __shared__ uint32_t part_max[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int part = warp % WPR, li = 32 * part + lane;
    const int nblk = (int)(K >> 4);
    const int ncol_pad = SWZ ? ((nblk + 3) & ~3) : nblk;
    const int64_t rows_iter = SWZ ? ((rows + 127) & ~(int64_t)127) : rows;
    // CTA-uniform loop over pairs of rows (the shared-memory fold synchronizes the CTA)
    for (int64_t r0 = (int64_t)blockIdx.x * 2; r0 < rows_iter; r0 += (int64_t)gridDim.x * 2) {
        const int64_t r = r0 + warp / WPR;
        const bool in_iter = r < rows_iter, real = r < rows;
        if (in_iter && !real) {  // swizzle padding rows
            for (int b = li; b < ncol_pad; b += 32 * WPR) store_sf(sf, SWZ, r, b, nblk, 0u);
        }
        const uint16_t* xr = x + r * ldx;
        uint4 va[BPL], vb[BPL];
        uint32_t bmax[BPL];
        uint32_t rmax = 0;
#pragma unroll
        for (int i = 0; i < BPL; ++i) {
            const int b = li + 32 * WPR * i;
            if (real && b < nblk) {
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
        float t = 0.0f;
        if (TMODE == 0) {
            rmax = __reduce_max_sync(0xFFFFFFFFu, rmax);
            if (lane == 0) part_max[warp] = rmax;
            __syncthreads();
            const int w0 = warp - part;
#pragma unroll
            for (int p = 0; p < WPR; ++p) rmax = max(rmax, part_max[w0 + p]);
            __syncthreads();
            t = __fdiv_rn(bf16mag_to_f32(rmax), kNvfp4ScaleDivisor);
            if (li == 0 && real) row_scale[r] = t;
        } else if (real) {
            t = __fdiv_rn(group_amax[r / rpg], kNvfp4ScaleDivisor);
        }
        if (!real) continue;
        const float six_t = __fmul_rn(6.0f, t), four_t = __fmul_rn(4.0f, t);
        uint2* crow = reinterpret_cast<uint2*>(codes + r * (K >> 1));
#pragma unroll
        for (int i = 0; i < BPL; ++i) {
            const int b = li + 32 * WPR * i;
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
    pdl_enter();
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
// Phase 1 (row copy): thread item = (row r, 16-byte chunk ch of 8 bf16), four
// lanes per 32-element block, straight from registers; the tile also goes to
// shared memory (256-byte rows, chunk ch of row r stored at
// ch ^ (((r >> 3) & 3) << 2)).
// Phase 2 (column copy): thread = (column quad q, row group g): it reads 8
// rows of 4 columns (columns 4q .. 4q+3, rows 8g .. 8g+7) with 8-byte loads.
// Warp w covers column quads 8 (w & 3) .. +7 and row groups 4 (w >> 2) .. +3,
// i.e. one MXFP8 block (32 rows) of 32 columns: the block maxima are folded
// over the 4 row groups by shuffles, and the permutation keeps the warp's 4
// rows on distinct banks.  Each thread writes 8 contiguous code bytes per
// column (32 contiguous bytes per block and column).  The block scale bytes
// of the tile's rows and of its columns each go through a 512-byte shared
// table and leave as one 32-bit word (4 consecutive blocks) per row or column.
constexpr int MX_TILE = 128;

BSQ_DEVICE int mx_chunk(int r, int ch) { return r * 16 + (ch ^ (((r >> 3) & 3) << 2)); }  // in 16-byte units

template <bool SWZ, bool ROW, bool COL>
__global__ void __launch_bounds__(512) k_mxfp8_rowcol(const uint16_t* __restrict__ x, int64_t rows, int64_t K,
                                                      int64_t ldx, uint8_t* __restrict__ row_codes,
                                                      uint8_t* __restrict__ row_sf, uint8_t* __restrict__ col_codes,
                                                      uint8_t* __restrict__ col_sf)
{
    pdl_enter();
    __shared__ __align__(16) uint4 tile[MX_TILE * 16];
    __shared__ uint8_t sfrow[MX_TILE][4];  // row scale bytes of the tile's 4 blocks per row
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row0 = (int64_t)blockIdx.y * MX_TILE, col0 = (int64_t)blockIdx.x * MX_TILE;
    const int64_t nsf_row = K >> 5, nsf_col = rows >> 5;
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int item = tid + 512 * i;
        const int r = item >> 4, ch = item & 15;
        const int64_t gr = row0 + r, gc = col0 + 8 * ch;
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (gr < rows && gc < K) v[i] = ldg_stream(x + gr * ldx + gc);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int item = tid + 512 * i;
        const int r = item >> 4, ch = item & 15;
        const int64_t gr = row0 + r, gc = col0 + 8 * ch;
        if (COL) tile[mx_chunk(r, ch)] = v[i];
        if (ROW) {
            uint32_t m = absmax_bf16x2(0u, v[i].x);
            m = absmax_bf16x2(m, v[i].y);
            m = absmax_bf16x2(m, v[i].z);
            m = absmax_bf16x2(m, v[i].w);
            m = fold_halves(m);
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            uint2 c = make_uint2(0u, 0u);
            uint32_t s = 0;
            if (m) {
                const int X = mx_exponent(m << 16);
                const float mul = mx_multiplier(X);
                s = (uint32_t)(X + 127);
                c.x = e4m3x4(__fmul_rn(bf16_lo(v[i].x), mul), __fmul_rn(bf16_hi(v[i].x), mul),
                             __fmul_rn(bf16_lo(v[i].y), mul), __fmul_rn(bf16_hi(v[i].y), mul));
                c.y = e4m3x4(__fmul_rn(bf16_lo(v[i].z), mul), __fmul_rn(bf16_hi(v[i].z), mul),
                             __fmul_rn(bf16_lo(v[i].w), mul), __fmul_rn(bf16_hi(v[i].w), mul));
            }
            const bool ok = gr < rows && gc < K;
            if (ok) *reinterpret_cast<uint2*>(row_codes + gr * K + gc) = c;
            if ((ch & 3) == 0) sfrow[r][ch >> 2] = (uint8_t)s;
        }
    }
    __syncthreads();
    if (ROW && tid >= 512 - MX_TILE) {  // one word of 4 block scales per row of the tile
        const int r = tid - (512 - MX_TILE);
        const int64_t gr = row0 + r, cb = col0 >> 5;
        if (gr < rows && col0 < K) {
            const uint32_t word = *reinterpret_cast<const uint32_t*>(sfrow[r]);
            if (SWZ || ((nsf_row & 3) == 0 && cb + 4 <= nsf_row)) {
                const int64_t o = SWZ ? sf_swizzled(gr, cb, (nsf_row + 3) >> 2) : gr * nsf_row + cb;
                *reinterpret_cast<uint32_t*>(row_sf + o) = word;
            } else {
                for (int j = 0; j < 4; ++j)
                    if (cb + j < nsf_row) row_sf[gr * nsf_row + cb + j] = (uint8_t)(word >> (8 * j));
            }
        }
    }
    if (!COL) return;
    __shared__ uint8_t sfcol[MX_TILE][4];  // column scale bytes of the tile's 4 blocks
    const int cs = lane & 7, gs = lane >> 3;
    const int q = 8 * (warp & 3) + cs;    // column quad: columns 4q .. 4q+3 of the tile
    const int g = 4 * (warp >> 2) + gs;   // row group: rows 8g .. 8g+7
    const int blk = warp >> 2;            // the tile's MXFP8 block these rows belong to
    const uint8_t* tb = reinterpret_cast<const uint8_t*>(tile);
    uint2 cv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 8 * g + i;
        cv[i] = *reinterpret_cast<const uint2*>(tb + 16 * mx_chunk(r, q >> 1) + 8 * (q & 1));
    }
    uint32_t m01 = 0u, m23 = 0u;  // bf16 magnitude maxima of columns (0, 1) and (2, 3)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        m01 = absmax_bf16x2(m01, cv[i].x);
        m23 = absmax_bf16x2(m23, cv[i].y);
    }
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {  // the other 3 row groups of the block
        m01 = __vmaxu2(m01, __shfl_xor_sync(0xFFFFFFFFu, m01, off));
        m23 = __vmaxu2(m23, __shfl_xor_sync(0xFFFFFFFFu, m23, off));
    }
    const int64_t gr = row0 + 8 * g;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t mc = ((c < 2 ? m01 : m23) >> (16 * (c & 1))) & 0xFFFFu;
        uint32_t w0 = 0u, w1 = 0u, sc = 0u;
        if (mc) {
            const int X = mx_exponent(mc << 16);
            const float mul = mx_multiplier(X);
            sc = (uint32_t)(X + 127);
            float f[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t w = c < 2 ? cv[i].x : cv[i].y;
                f[i] = __fmul_rn((c & 1) ? bf16_hi(w) : bf16_lo(w), mul);
            }
            w0 = e4m3x4(f[0], f[1], f[2], f[3]);
            w1 = e4m3x4(f[4], f[5], f[6], f[7]);
        }
        const int64_t gc = col0 + 4 * q + c;
        if (gc < K && gr < rows) *reinterpret_cast<uint2*>(col_codes + gc * rows + gr) = make_uint2(w0, w1);
        if (gs == 0) sfcol[4 * q + c][blk] = (uint8_t)sc;
    }
    __syncthreads();
    if (tid < MX_TILE) {  // one word of 4 block scales per column of the tile
        const int64_t gc = col0 + tid, cb = row0 >> 5;
        if (gc < K && row0 < rows) {
            const uint32_t word = *reinterpret_cast<const uint32_t*>(sfcol[tid]);
            if (SWZ || ((nsf_col & 3) == 0 && cb + 4 <= nsf_col)) {
                const int64_t o = SWZ ? sf_swizzled(gc, cb, (nsf_col + 3) >> 2) : gc * nsf_col + cb;
                *reinterpret_cast<uint32_t*>(col_sf + o) = word;
            } else {
                for (int j = 0; j < 4; ++j)
                    if (cb + j < nsf_col) col_sf[gc * nsf_col + cb + j] = (uint8_t)(word >> (8 * j));
            }
        }
    }
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
// A launch with programmatic dependent launch allowed (pdl): the grid may be
// launched while the previous one in the stream drains, and its kernel waits
// for it in pdl_enter() before touching memory.  The standalone quantizer
// entry points use it, so back-to-back calls overlap one call's tail with the
// next one's launch; in the MoE forward the light kernels use it and the
// GEMMs launch plainly (their persistent CTAs need the SMs to themselves).
template <typename... KArgs, typename... Args>
static void launch_ks(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, bool pdl, cudaStream_t st,
                      Args... args)
{
    if (!pdl) {
        kernel<<<grid, block, smem, st>>>(args...);
        return;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
template <typename... KArgs, typename... Args>
static void launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, bool pdl, cudaStream_t st, Args... args)
{
    launch_ks(kernel, grid, block, 0, pdl, st, args...);
}

static int grid_for(int64_t warps_needed, int sms)
{
    const int64_t blocks = (warps_needed + 7) / 8;
    const int64_t cap = (int64_t)sms * 16;
    return (int)std::max<int64_t>(1, std::min<int64_t>(blocks, cap));
}

template <bool F46, bool SWZ, int TM>
static void launch_rows_t(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx, uint8_t* codes, uint8_t* sf,
                          float* rs, const float* gam, int64_t rpg, int sms, bool pdl, cudaStream_t st)
{
    const int nblk = (int)(K >> 4);
    const int64_t rows_iter = SWZ ? ((rows + 127) & ~(int64_t)127) : rows;
    const int grid = grid_for(rows_iter, sms);
    if (nblk == 48)  // e.g. K = 768: a half-warp per row, 3 blocks per lane
        launch_k(k_nvfp4_rows<3, F46, SWZ, TM, 16>, dim3(grid_for((rows_iter + 1) / 2, sms)), dim3(256), pdl, st, x,
                 rows, K, ldx, codes, sf, rs, gam, rpg);
    else if (nblk <= 32)
        launch_k(k_nvfp4_rows<1, F46, SWZ, TM>, dim3(grid), dim3(256), pdl, st, x, rows, K, ldx, codes, sf, rs, gam, rpg);
    else if (nblk <= 64)
        launch_k(k_nvfp4_rows<2, F46, SWZ, TM>, dim3(grid), dim3(256), pdl, st, x, rows, K, ldx, codes, sf, rs, gam, rpg);
    else if (nblk <= 128)  // ~70 registers a thread: CTAs of 4 warps fill an SM (28 warps) better than of 8 (24)
        launch_k(k_nvfp4_rows<4, F46, SWZ, TM>, dim3(2 * grid), dim3(128), pdl, st, x, rows, K, ldx, codes, sf, rs, gam,
                 rpg);
    else if (nblk <= 512)
        launch_k(k_nvfp4_rows_wide<F46, SWZ, TM>, dim3(grid_for(rows_iter * 4, sms)), dim3(256), pdl, st, x, rows, K,
                 ldx, codes, sf, rs, gam, rpg);
    else
        launch_k(k_nvfp4_rows_long<F46, SWZ, TM>, dim3(grid), dim3(256), pdl, st, x, rows, K, ldx, codes, sf, rs, gam,
                 rpg);
}

void launch_nvfp4_rows(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx, uint8_t* codes, uint8_t* sf,
                       float* row_scale, const float* group_amax, int64_t rpg, bool four_six, bool swz, int sms,
                       bool pdl, cudaStream_t st)
{
    const bool per_group = group_amax != nullptr;
#define BSQ_ROWS(F, S, T) launch_rows_t<F, S, T>(x, rows, K, ldx, codes, sf, row_scale, group_amax, rpg, sms, pdl, st)
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
#define BSQ_MX(S, R, C) launch_k(k_mxfp8_rowcol<S, R, C>, grid, dim3(512), true, st, x, rows, K, ldx, rc, rs, cc, cs)
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

// ---------------------------------------------------------------- RHT + NVFP4
// Per-token NVFP4 of a 32-point random Hadamard transform of each row
// ("End-to-End 4-Bit Training", section "第三个决定": the transform spreads
// outliers over their group before block quantization).  Per group of 32
// consecutive elements, y = H32 (s . x) with the Sylvester matrix unnormalized,
// in binary32 by the butterfly h = 1, 2, 4, 8, 16; s = the 32 bits of word 0
// of Philox4x32-10(seed, (0, 0, 2, 0)) (bit j set: s_j = -1).  Two warps per
// row: of each chunk of 128 blocks (2048 elements), warp h takes blocks
// 64 h + lane + 32 i (i < 2), so a block's group partner (block b ^ 1) sits in
// lane l ^ 1 of the same warp at the same register slot: stages 1-8 run in
// registers, stage 16 is one shuffle.  The row maximum is folded over the two
// warps in shared memory.  Rows of up to 128 blocks are quantized from
// registers (32 values a lane: ~64 registers, 32 warps an SM); longer rows
// take two passes over their chunks (the transformed row's maximum, then the
// encode).  One warp per whole row held 64 values a lane at 128 registers
// and 16 warps an SM, and took 37.5 us on 16384 x 2048; this form takes
// 35.2 us with four CTAs an SM (64 registers, a small spill) and 35.9 us with
// three, so occupancy is not what bounds it.
namespace {

// The sign flips of this lane's 16 elements (its block's half of the
// group) as XOR masks on the 8 packed bf16 words: element 2 j is the low half
// of word j (sign bit 15), element 2 j + 1 the high half (bit 31).
BSQ_DEVICE void rht_sign_masks(uint32_t signs, int lane, uint32_t (&m)[8])
{
    const uint32_t sg = (lane & 1) ? (signs >> 16) : signs;
#pragma unroll
    for (int j = 0; j < 8; ++j) m[j] = (((sg >> (2 * j)) & 1u) << 15) | (((sg >> (2 * j + 1)) & 1u) << 31);
}

BSQ_DEVICE void rht_blocks(const uint16_t* __restrict__ xr, int nblk, int b0, int lane, const uint32_t (&sm)[8],
                           float (&v)[2][16])
{
    // the cross-lane stage: the even lane of a pair keeps v + o, the odd lane
    // o - v; fma(+-1, v, o) rounds the same sum or difference once
    const float pm = (lane & 1) ? -1.0f : 1.0f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int b = b0 + lane + 32 * i;
        uint4 a = make_uint4(0u, 0u, 0u, 0u), c = make_uint4(0u, 0u, 0u, 0u);
        if (b < nblk) {
            a = ldg_stream(xr + 16 * b);
            c = ldg_stream(xr + 16 * b + 8);
        }
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t ws = w[j] ^ sm[j];  // s . x: bf16 negation is a sign-bit flip
            v[i][2 * j] = bf16_lo(ws);
            v[i][2 * j + 1] = bf16_hi(ws);
        }
#pragma unroll
        for (int h = 1; h < 16; h <<= 1)
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if ((j & h) == 0) {
                    const float p = v[i][j], q = v[i][j + h];
                    v[i][j] = __fadd_rn(p, q);
                    v[i][j + h] = __fsub_rn(p, q);
                }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float o = __shfl_xor_sync(0xFFFFFFFFu, v[i][j], 1);
            v[i][j] = __fmaf_rn(pm, v[i][j], o);
        }
    }
}

template <bool SWZ>
__global__ void __launch_bounds__(256, 4) k_nvfp4_rht(const uint16_t* __restrict__ x, int64_t rows, int64_t K, int64_t ldx,
                                                   uint64_t seed, uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                   float* __restrict__ row_scale)
{
    pdl_enter();
    __shared__ float s_max[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, half = warp & 1;
    const int nblk = (int)(K >> 4);
    const int ncol_pad = SWZ ? ((nblk + 3) & ~3) : nblk;
    const int64_t nct = (ncol_pad + 3) >> 2;
    const int64_t rows_iter = SWZ ? ((rows + 127) & ~(int64_t)127) : rows;
    const uint32_t signs = philox4x32_10(make_uint4(0u, 0u, 2u, 0u), (uint32_t)seed, (uint32_t)(seed >> 32)).x;
    uint32_t sm[8];
    rht_sign_masks(signs, lane, sm);
    // CTA-uniform loop over groups of 4 rows (the shared-memory fold synchronizes the CTA)
    for (int64_t r0 = (int64_t)blockIdx.x * 4; r0 < rows_iter; r0 += (int64_t)gridDim.x * 4) {
        const int64_t r = r0 + (warp >> 1);
        const bool real = r < rows;
        const uint16_t* xr = x + r * ldx;
        float v[2][16];
        float amax = 0.0f;
        for (int c0 = 0; c0 < nblk; c0 += 128) {  // one chunk for rows of up to 128 blocks
            if (real) rht_blocks(xr, nblk, c0 + 64 * half, lane, sm, v);
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 16; ++j) amax = real ? fmaxf(amax, fabsf(v[i][j])) : 0.0f;
        }
        amax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(amax)));  // non-negative: bit order
        if (lane == 0) s_max[warp] = amax;
        __syncthreads();
        amax = fmaxf(s_max[warp & ~1], s_max[warp | 1]);
        __syncthreads();
        if (r >= rows_iter) continue;
        if (!real) {  // swizzle padding rows: zero scale factors
            for (int b = 32 * half + lane; b < ncol_pad; b += 64) sf[sf_swizzled(r, b, nct)] = 0u;
            continue;
        }
        const float t = __fdiv_rn(amax, kNvfp4ScaleDivisor);
        if (lane == 0 && half == 0) row_scale[r] = t;
        const float six_t = __fmul_rn(6.0f, t);
        uint2* crow = reinterpret_cast<uint2*>(codes + r * (K >> 1));
        for (int c0 = 0; c0 < nblk; c0 += 128) {
            if (nblk > 128) rht_blocks(xr, nblk, c0 + 64 * half, lane, sm, v);  // second pass: transform again
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int b = c0 + 64 * half + lane + 32 * i;
                if (b >= nblk) {
                    if (SWZ && b < ncol_pad) sf[sf_swizzled(r, b, nct)] = 0u;
                    continue;
                }
                uint2 c = make_uint2(0u, 0u);
                uint32_t sfb = 0u;
                if (t != 0.0f) {
                    float ab = 0.0f;
#pragma unroll
                    for (int j = 0; j < 16; ++j) ab = fmaxf(ab, fabsf(v[i][j]));
                    const BlockScale bs = nvfp4_block_scale(ab, six_t, t);
                    c = encode16(v[i], bs.enc);
                    sfb = bs.sf;
                }
                crow[b] = c;
                sf[SWZ ? sf_swizzled(r, b, nct) : r * nblk + b] = (uint8_t)sfb;
            }
        }
    }
}

}  // namespace

void launch_nvfp4_rht(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx, uint64_t seed, uint8_t* codes,
                      uint8_t* sf, float* row_scale, bool swz, int sms, cudaStream_t st)
{
    const int64_t rows_iter = swz ? ((rows + 127) & ~(int64_t)127) : rows;
    const dim3 grid((unsigned)std::max<int64_t>(1, std::min<int64_t>((rows_iter + 3) / 4, (int64_t)sms * 8)));
    if (swz)
        launch_k(k_nvfp4_rht<true>, grid, dim3(256), true, st, x, rows, K, ldx, seed, codes, sf, row_scale);
    else
        launch_k(k_nvfp4_rht<false>, grid, dim3(256), true, st, x, rows, K, ldx, seed, codes, sf, row_scale);
}

// ---------------------------------------------------------------- 2-D NVFP4
// One E4M3 scale per 16 x 16 tile and one FP32 scale per tensor ("End-to-End
// 4-Bit Training", section "第二个决定": square block scales are the same
// before and after the transpose, so the transposed backward operand is the
// same codes and scales rearranged, with no requantization; the price is 256
// values under one scale).
// Pass 1, the tensor maximum: grid-stride 16-byte loads, 8 in flight per
// thread, folded per warp and per CTA, one atomic per CTA.
// Pass 2: a CTA takes 128 rows x 128 columns; warp w the 16-row strip w of
// it.  Lanes 4p .. 4p + 3 take 4 columns each of tile p over its 16 rows
// (8-byte loads: every load instruction reads 256 contiguous bytes of a row,
// and 32 registers hold the data); the tile maximum (packed bf16 |max|) is
// folded over the four lanes.  The row-major codes leave as 2 bytes per lane
// and row (64 contiguous bytes per instruction).  For the transposed codes
// (8 bytes = 16 rows per column and strip) the code words of rows 4g, 4g + 2
// and 4g + 1, 4g + 3 are packed in pairs and interleaved by nibble, which
// puts each column's row pairs in bytes; one byte permute per column and 8
// rows gathers them.  They meet in shared memory, in 72-byte rows with the
// strip slot rotated by column so that a warp's 256 bytes take the minimum
// two wavefronts; two threads then write each column's 64 bytes (the CTA's
// 128 rows) of the transposed operand, 32 bytes each.
namespace {

__global__ void __launch_bounds__(256) k_tensor_amax(const uint16_t* __restrict__ x, int64_t n8,
                                                     unsigned int* __restrict__ amax_bits)
{
    __shared__ uint32_t s_m[8];
    uint32_t m = 0;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i < n8; i += 8 * stride) {  // 8 loads in flight, the tail predicated
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            v[u] = i + u * stride < n8 ? ldg_stream(x + 8 * (i + u * stride)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            uint32_t a = absmax_bf16x2(0u, v[u].x);
            a = absmax_bf16x2(a, v[u].y);
            a = absmax_bf16x2(a, v[u].z);
            a = absmax_bf16x2(a, v[u].w);
            m = max(m, fold_halves(a));
        }
    }
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0) s_m[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = max(m, s_m[w]);
        if (m) atomicMax(amax_bits, m << 16);
    }
}

// Four binary32 values -> four E2M1 codes in the low 16 bits (element i in
// nibble i), RNE satfinite.
BSQ_DEVICE uint32_t e2m1x4_16(float v0, float v1, float v2, float v3)
{
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1;\n\t.reg .b16 h;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "mov.b16 h, {b0, b1};\n\tcvt.u32.u16 %0, h;\n\t}"
        : "=r"(r)
        : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
    return r;
}

template <bool T_OUT>
__global__ void __launch_bounds__(256) k_nvfp4_2d(const uint16_t* __restrict__ x, int64_t rows, int64_t K,
                                                  const float* __restrict__ tscale, uint8_t* __restrict__ codes,
                                                  uint8_t* __restrict__ sf, uint8_t* __restrict__ codes_t,
                                                  uint8_t* __restrict__ sf_t, bool vec32_t)
{
    pdl_enter();
    __shared__ uint2 s_t[128][9];   // [column of the CTA tile][rotated strip slot], one slot of padding
    __shared__ uint8_t s_sf[8][8];  // [column tile][row strip]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ctiles = (K + 127) >> 7;
    const int64_t nblk = ((rows + 127) >> 7) * ctiles;
    const float t = __ldg(tscale);
    const float six_t = __fmul_rn(6.0f, t);
    for (int64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
        const int64_t R0 = (blk / ctiles) << 7, C0 = (blk % ctiles) << 7;
        const int64_t r0 = R0 + 16 * warp, c0 = C0 + 4 * lane;  // this lane's first row and column
        const bool valid = r0 < rows && c0 < K;                  // K % 16 == 0: the lanes of a tile agree
        uint2 v[16];
        uint32_t m2 = 0;  // packed bf16 max of |x| (sign bits meaningless until masked)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            v[i] = valid ? __ldcs(reinterpret_cast<const uint2*>(x + (r0 + i) * K + c0)) : make_uint2(0u, 0u);
            asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(v[i].x));
            asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(v[i].y));
        }
        uint32_t m = fold_halves(m2 & 0x7FFF7FFFu);
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
        uint32_t sfb = 0u;
        float enc = 0.0f;
        if (t != 0.0f) {
            const BlockScale bs = nvfp4_block_scale(bf16mag_to_f32(m), six_t, t);
            sfb = bs.sf;
            enc = bs.enc;
        }
        uint32_t w[16];  // 4 codes (16 bits) of row i
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            w[i] = (t != 0.0f) ? e2m1x4_16(__fmul_rn(bf16_lo(v[i].x), enc), __fmul_rn(bf16_hi(v[i].x), enc),
                                           __fmul_rn(bf16_lo(v[i].y), enc), __fmul_rn(bf16_hi(v[i].y), enc))
                               : 0u;
            if (valid) *reinterpret_cast<uint16_t*>(codes + (r0 + i) * (K >> 1) + (c0 >> 1)) = (uint16_t)w[i];
        }
        if (valid && (lane & 3) == 0) sf[(r0 >> 4) * (K >> 4) + (c0 >> 4)] = (uint8_t)sfb;
        if constexpr (T_OUT) {
            // rows 4g, 4g + 1 (bytes 0, 1) and 4g + 2, 4g + 3 (bytes 2, 3) of
            // columns 0, 2 (ev) and 1, 3 (od): row 4g + 2k in the low nibble
            uint32_t ev[4], od[4];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const uint32_t wa = __byte_perm(w[4 * g], w[4 * g + 2], 0x5410u);
                const uint32_t wb = __byte_perm(w[4 * g + 1], w[4 * g + 3], 0x5410u);
                ev[g] = (wa & 0x0F0F0F0Fu) | ((wb << 4) & 0xF0F0F0F0u);
                od[g] = ((wa >> 4) & 0x0F0F0F0Fu) | (wb & 0xF0F0F0F0u);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t* q = (j & 1) ? od : ev;
                const uint32_t sel = (j & 2) ? 0x7531u : 0x6420u;  // columns 2, 3: the odd bytes
                const int col = 4 * lane + j;
                s_t[col][(warp + (col >> 4)) & 7] = make_uint2(__byte_perm(q[0], q[1], sel), __byte_perm(q[2], q[3], sel));
            }
            if ((lane & 3) == 0) s_sf[lane >> 2][warp] = (uint8_t)sfb;
            __syncthreads();
            // column C0 + c of x = row C0 + c of the transposed operand; thread 2c + h writes
            // its row strips 4h .. 4h + 3 (32 bytes)
            const int c = threadIdx.x >> 1, h = threadIdx.x & 1;
            const int64_t col = C0 + c;
            const int nst = (int)(((rows - R0) >> 4) < 8 ? ((rows - R0) >> 4) : 8);  // row strips present
            if (col < K) {
                uint2 q[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) q[k] = s_t[c][(4 * h + k + (c >> 4)) & 7];
                uint2* dst = reinterpret_cast<uint2*>(codes_t + col * (rows >> 1) + (R0 >> 1)) + 4 * h;
                if (nst == 8 && vec32_t) {
                    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(q[0].x),
                                 "r"(q[0].y), "r"(q[1].x), "r"(q[1].y), "r"(q[2].x), "r"(q[2].y), "r"(q[3].x),
                                 "r"(q[3].y)
                                 : "memory");
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (4 * h + k < nst) dst[k] = q[k];
                }
            }
            if (threadIdx.x < 64) {
                const int ct = threadIdx.x >> 3, k = threadIdx.x & 7;
                if (k < nst && C0 + 16 * ct < K) sf_t[((C0 >> 4) + ct) * (rows >> 4) + (R0 >> 4) + k] = s_sf[ct][k];
            }
            __syncthreads();
        }
    }
}

}  // namespace

cudaError_t launch_nvfp4_2d(const uint16_t* x, int64_t rows, int64_t K, uint8_t* codes, uint8_t* sf,
                            uint8_t* codes_t, uint8_t* sf_t, float* tscale, int sms, cudaStream_t st)
{
    cudaError_t err = cudaMemsetAsync(tscale, 0, sizeof(float), st);
    if (err != cudaSuccess) return err;
    const int64_t n8 = rows * K / 8;
    k_tensor_amax<<<(unsigned)std::max<int64_t>(1, std::min<int64_t>((n8 + 255) / 256, (int64_t)sms * 8)), 256, 0,
                    st>>>(x, n8, reinterpret_cast<unsigned int*>(tscale));
    launch_group_finalize(tscale, 1, st);
    const int64_t nblk = ((rows + 127) >> 7) * ((K + 127) >> 7);
    const int64_t grid = std::min<int64_t>(nblk, (int64_t)sms * 8);
    if (grid <= 0) return cudaSuccess;
    const bool vec32_t = codes_t && (reinterpret_cast<uintptr_t>(codes_t) % 32 == 0) && ((rows >> 1) % 32 == 0);
    if (codes_t)
        launch_k(k_nvfp4_2d<true>, dim3((unsigned)grid), dim3(256), true, st, x, rows, K, (const float*)tscale, codes,
                 sf, codes_t, sf_t, vec32_t);
    else
        launch_k(k_nvfp4_2d<false>, dim3((unsigned)grid), dim3(256), true, st, x, rows, K, (const float*)tscale, codes,
                 sf, (uint8_t*)nullptr, (uint8_t*)nullptr, false);
    return cudaSuccess;
}

// ---------------------------------------------------------------- dequantize
// BF16 operands for the dequantized backward mode ("LMSYS Drops Miles ...",
// "Recipe 2: Per-token NVFP4 for MoE experts": the backward GEMMs run in BF16
// on BF16 dequantizations of the exact low-precision forward operands).
// y = bf16_rn(rn(rn(e2m1 * sf) * t)) with t the row's (per-token) or the
// row's group's (per-expert) FP32 scale.  Bound by HBM writes: per element
// 0.5 B of codes and 1/16 B of scale factor in, 2 B out.  One warp per row;
// lane l takes the row's 16-element blocks l, l + 32, l + 64, l + 96 (all
// loads first, then the dequantization and the stores), so every store
// instruction of the warp writes 1 KB of the row contiguously and every code
// load reads 256 contiguous bytes.  Rows beyond the first wave of warps are
// taken grid-stride.  (Four consecutive blocks per thread, 128-byte strided
// stores, ran at 21.5 us on 16384 x 2048 against 17.1 us.)
namespace {

BSQ_DEVICE void store_bf16x16(uint16_t* dst, const uint32_t (&w)[8], bool vec32)
{
    if (vec32) {
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                     : "memory");
    } else {
        uint4* q = reinterpret_cast<uint4*>(dst);
        q[0] = make_uint4(w[0], w[1], w[2], w[3]);
        q[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

BSQ_DEVICE uint32_t bf16x2_rn(float lo, float hi)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

template <bool SWZ>
__global__ void __launch_bounds__(256) k_dequant_nvfp4(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ sf,
                                                       const float* __restrict__ scale, int64_t rows, int K,
                                                       int64_t group_rows, uint16_t* __restrict__ y, int64_t ldy,
                                                       bool vec32)
{
    pdl_enter();
    const int kb = K >> 4;  // 16-element blocks per row
    const int lane = threadIdx.x & 31;
    const int64_t ncol_tiles = (kb + 3) >> 2;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows; row += nwarps) {
        const float t = __ldg(scale + (group_rows == 1 ? row : row / group_rows));
        const uint8_t* crow = codes + row * (int64_t)(K >> 1);
        uint16_t* yrow = y + row * ldy;
        for (int j0 = 0; j0 < kb; j0 += 128) {
            uint2 w[4];
            uint32_t sb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = j0 + lane + 32 * i;
                if (c < kb) {
                    w[i] = __ldg(reinterpret_cast<const uint2*>(crow + (int64_t)c * 8));
                    sb[i] = __ldg(sf + (SWZ ? sf_swizzled(row, c, ncol_tiles) : row * kb + c));
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = j0 + lane + 32 * i;
                if (c < kb) {
                    float d[16];
                    e2m1x8_dequant(w[i].x, sb[i], t, *reinterpret_cast<float(*)[8]>(d));
                    e2m1x8_dequant(w[i].y, sb[i], t, *reinterpret_cast<float(*)[8]>(d + 8));
                    uint32_t o[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) o[j] = bf16x2_rn(d[2 * j], d[2 * j + 1]);
                    store_bf16x16(yrow + (int64_t)c * 16, o, vec32);
                }
            }
        }
    }
}

}  // namespace

void launch_dequant_nvfp4(const uint8_t* codes, const uint8_t* sf, const float* scale, int64_t rows, int64_t K,
                          int64_t group_rows, uint16_t* y, int64_t ldy, bool swz, int sms, cudaStream_t st)
{
    const int64_t grid = std::min<int64_t>((rows + 7) / 8, (int64_t)sms * 16);  // 8 warps (rows) per CTA
    if (grid <= 0) return;
    const bool vec32 = (reinterpret_cast<uintptr_t>(y) % 32 == 0) && (ldy % 16 == 0);
    if (swz)
        launch_k(k_dequant_nvfp4<true>, dim3((unsigned)grid), dim3(256), true, st, codes, sf, scale, rows, (int)K,
                 group_rows, y, ldy, vec32);
    else
        launch_k(k_dequant_nvfp4<false>, dim3((unsigned)grid), dim3(256), true, st, codes, sf, scale, rows, (int)K,
                 group_rows, y, ldy, vec32);
}

}  // namespace bsq
