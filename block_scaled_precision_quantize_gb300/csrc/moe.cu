// moe.cu -- the non-GEMM steps of the MoE expert forward: routing
// (count / padded scan / stable slot assignment), per-token NVFP4
// quantization scattered into the routed slots, and the weighted combine.
//
// Dispatch ("End-to-End 4-Bit Training" summary, section "第三个决定"): tokens
// travel to their experts already quantized.  Each expert's rows form one
// segment of the routed matrix, padded to a multiple of 128 rows (the GEMM
// tile height); inside a segment rows are in ascending (token, k) order, so
// the layout is deterministic.
#include "common.cuh"
#include "kernels.h"

namespace bsq {

constexpr int RT_CHUNK = 512;  // routed pairs per histogram chunk

// Phase A: per-chunk expert histograms -> hist[chunk][E].  Also clears the
// ticket counter of phase B (stream order puts this before phase B).
__global__ void __launch_bounds__(256) k_route_hist(const int32_t* __restrict__ ids, int64_t n, int32_t E,
                                                    int32_t* __restrict__ hist, int32_t* __restrict__ ticket,
                                                    int32_t* dev_status)
{
    pdl_enter();
    extern __shared__ int32_t sh[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0;
    __syncthreads();
    const int64_t i0 = (int64_t)blockIdx.x * RT_CHUNK, i1 = min(n, i0 + RT_CHUNK);
    for (int64_t i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
        const int32_t e = __ldg(ids + i);
        if (e >= 0 && e < E) atomicAdd(sh + e, 1);
        else report(dev_status, BSQ_DEV_BAD_EXPERT);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(int64_t)blockIdx.x * E + e] = sh[e];
}

// Exclusive prefix of v over the 256 threads of a CTA; *total gets the sum.
__device__ __forceinline__ int32_t block_exclusive_scan256(int32_t v, int32_t* warp_sums, int32_t* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += u;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    int32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const int32_t ws = warp_sums[w];
        before += (w < warp) ? ws : 0;
        all += ws;
    }
    __syncthreads();
    *total = all;
    return before + incl - v;
}

// Phase B: CTA e turns column e of hist into its exclusive prefix over the
// chunks (in place) and writes counts[e]; the last CTA to finish (ticket)
// then lays out the segments: offsets[e] = sum over e' < e of counts[e']
// rounded up to 128, offsets[E] = the total.
__global__ void __launch_bounds__(256) k_route_scan(int32_t* __restrict__ hist, int32_t nchunks, int32_t E,
                                                    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ ticket)
{
    pdl_enter();
    __shared__ int32_t warp_sums[8];
    __shared__ bool last;
    const int e = blockIdx.x;
    int32_t carry = 0;
    for (int c0 = 0; c0 < nchunks; c0 += 256) {
        const int c = c0 + threadIdx.x;
        const int32_t v = c < nchunks ? hist[(int64_t)c * E + e] : 0;
        int32_t total;
        const int32_t ex = block_exclusive_scan256(v, warp_sums, &total);
        if (c < nchunks) hist[(int64_t)c * E + e] = carry + ex;
        carry += total;
    }
    if (threadIdx.x == 0) {
        counts[e] = carry;
        __threadfence();
        last = atomicAdd(ticket, 1) == E - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    int32_t base = 0;
    for (int e0 = 0; e0 < E; e0 += 256) {
        const int ee = e0 + threadIdx.x;
        const int32_t padded = ee < E ? ((__ldcg(counts + ee) + 127) & ~127) : 0;
        int32_t total;
        const int32_t ex = block_exclusive_scan256(padded, warp_sums, &total);
        if (ee < E) offsets[ee] = base + ex;
        base += total;
    }
    if (threadIdx.x == 0) {
        offsets[E] = base;
        *ticket = 0;
    }
}

// Phase C, E <= RT_CTA_MAX_E: one CTA of 256 threads per chunk, two rounds of
// 256 pairs.  In a round, pair i goes to thread i; lanes of a warp routed to
// the same expert are ranked with __match_any_sync, the warps' per-expert
// counts go to shared memory, and a pair's slot is its expert's running fill
// + the counts of the earlier warps + its rank in the warp: the ascending
// (token, k) order of the single-warp walk below, in one pass per round.
constexpr int RT_CTA_MAX_E = 512;
__global__ void __launch_bounds__(256) k_route_assign_cta(const int32_t* __restrict__ ids, int64_t n, int32_t E,
                                                          const int32_t* __restrict__ hist,
                                                          const int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ slot_of, int32_t* __restrict__ row_src)
{
    pdl_enter();
    __shared__ int32_t fill[RT_CTA_MAX_E];
    __shared__ int32_t cnt[8][RT_CTA_MAX_E];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += 256) fill[e] = offsets[e] + hist[(int64_t)blockIdx.x * E + e];
    const int64_t i0 = (int64_t)blockIdx.x * RT_CHUNK, i1 = min(n, i0 + RT_CHUNK);
    for (int64_t base = i0; base < i1; base += 256) {
        for (int j = tid; j < 8 * E; j += 256) cnt[j / E][j % E] = 0;
        __syncthreads();
        const int64_t i = base + tid;
        const bool valid = i < i1;
        int32_t e = valid ? __ldg(ids + i) : -1;
        if (e >= E) e = -1;
        const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
        const int rank = __popc(same & ((1u << lane) - 1u));
        if (e >= 0 && rank == 0) cnt[warp][e] = __popc(same);
        __syncthreads();
        int32_t slot = -1;
        if (e >= 0) {
            int32_t before = 0;
            for (int w = 0; w < warp; ++w) before += cnt[w][e];
            slot = fill[e] + before + rank;
            row_src[slot] = (int32_t)i;
        }
        if (valid) slot_of[i] = slot;
        __syncthreads();
        for (int ee = tid; ee < E; ee += 256) {
            int32_t tot = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) tot += cnt[w][ee];
            fill[ee] += tot;
        }
        __syncthreads();
    }
}

// Phase C: one warp per chunk walks its pairs in order, 32 at a time; lanes
// routed to the same expert are ranked with __match_any_sync.
__global__ void __launch_bounds__(32) k_route_assign(const int32_t* __restrict__ ids, int64_t n, int32_t E,
                                                     const int32_t* __restrict__ hist,
                                                     const int32_t* __restrict__ offsets,
                                                     int32_t* __restrict__ slot_of, int32_t* __restrict__ row_src)
{
    pdl_enter();
    extern __shared__ int32_t fill[];
    const int lane = threadIdx.x;
    for (int e = lane; e < E; e += 32) fill[e] = offsets[e] + hist[(int64_t)blockIdx.x * E + e];
    __syncwarp();
    const int64_t i0 = (int64_t)blockIdx.x * RT_CHUNK, i1 = min(n, i0 + RT_CHUNK);
    for (int64_t base = i0; base < i1; base += 32) {
        const int64_t i = base + lane;
        const bool valid = i < i1;
        int32_t e = valid ? __ldg(ids + i) : -1;
        if (e >= E) e = -1;
        const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
        const int rank = __popc(same & ((1u << lane) - 1u));
        int32_t slot = -1;
        if (valid && e >= 0) {
            slot = fill[e] + rank;
            row_src[slot] = (int32_t)i;
        }
        if (valid) slot_of[i] = slot;
        __syncwarp();
        if (e >= 0 && rank == 0) fill[e] += __popc(same);
        __syncwarp();
    }
}

// Per-token NVFP4 quantization of x, written to every routed slot of the
// token (one warp per token, lane l owns 16-blocks l, l+32, ...).
// WPR warps share a token (wide rows: a row of 448 blocks at 4 blocks per
// lane instead of 16 keeps the registers, and so the occupancy, reasonable);
// a CTA of 8 warps takes 8 / WPR tokens per step and the row maximum is folded
// across the token's warps in shared memory.  Lane l of part p of a token owns
// blocks 32 p + l + 32 WPR i.
template <int BPL, bool FOUR_SIX, int WPR = 1>
__global__ void __launch_bounds__(256) k_quant_scatter(const uint16_t* __restrict__ x, int64_t T, int64_t H,
                                                       int32_t topk, const int32_t* __restrict__ slot_of,
                                                       const int32_t* __restrict__ offsets,
                                                       const int32_t* __restrict__ counts, int32_t E,
                                                       uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                       float* __restrict__ scale, int32_t* __restrict__ row_src,
                                                       int64_t cap)
{
    pdl_enter();
    const int TPC = (int)(blockDim.x >> 5) / WPR;  // tokens per CTA step (one per WPR warps)
    __shared__ uint32_t part_max[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int part = warp % WPR, li = 32 * part + lane;
    const int nblk = (int)(H >> 4);
    const int64_t ncol_tiles = (nblk + 3) >> 2;
    // The padding rows of every expert segment (from its last routed row up to
    // the next 128-row boundary) get scale 0 and all-zero scale factors, so the
    // GEMM's padding rows are exact zeros, and row_src -1: one expert per CTA,
    // one 4-byte scale-factor word per thread step.  The CTA after the last
    // expert marks the capacity past the last segment (row_src -1).
    for (int e = blockIdx.x; e <= E; e += gridDim.x) {
        if (e == E) {
            for (int64_t r = (int64_t)__ldg(offsets + E) + threadIdx.x; r < cap; r += blockDim.x) row_src[r] = -1;
            continue;
        }
        const int64_t p0 = (int64_t)__ldg(offsets + e) + __ldg(counts + e), p1 = __ldg(offsets + e + 1);
        for (int64_t i = threadIdx.x; i < (p1 - p0) * ncol_tiles; i += blockDim.x) {
            const int64_t r = p0 + i / ncol_tiles, wd = i % ncol_tiles;
            *reinterpret_cast<uint32_t*>(sf + sf_swizzled(r, 4 * wd, ncol_tiles)) = 0u;
            if (wd == 0) {
                scale[r] = 0.0f;
                row_src[r] = -1;
            }
        }
    }
    // CTA-uniform loop (the shared-memory fold below synchronizes the CTA)
    for (int64_t t0 = (int64_t)blockIdx.x * TPC; t0 < T; t0 += (int64_t)gridDim.x * TPC) {
        const int64_t t = t0 + warp / WPR;
        const bool real = t < T;
        const uint16_t* xr = x + t * H;
        uint4 va[BPL], vb[BPL];
        uint32_t bmax[BPL];
        uint32_t rmax = 0;
#pragma unroll
        for (int i = 0; i < BPL; ++i) {
            const int b = li + 32 * WPR * i;
            if (real && b < nblk) {
                asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(va[i].x), "=r"(va[i].y), "=r"(va[i].z), "=r"(va[i].w) : "l"(xr + 16 * b));
                asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(vb[i].x), "=r"(vb[i].y), "=r"(vb[i].z), "=r"(vb[i].w) : "l"(xr + 16 * b + 8));
            } else {
                va[i] = vb[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int i = 0; i < BPL; ++i) {
            uint32_t m = 0;
            const uint32_t w[8] = {va[i].x, va[i].y, va[i].z, va[i].w, vb[i].x, vb[i].y, vb[i].z, vb[i].w};
#pragma unroll
            for (int j = 0; j < 8; ++j) m = absmax_bf16x2(m, w[j]);
            bmax[i] = fold_halves(m);
            rmax = max(rmax, bmax[i]);
        }
        rmax = __reduce_max_sync(0xFFFFFFFFu, rmax);
        if (WPR > 1) {
            if (lane == 0) part_max[warp] = rmax;
            __syncthreads();
            const int w0 = warp - part;
#pragma unroll
            for (int p = 0; p < WPR; ++p) rmax = max(rmax, part_max[w0 + p]);
            __syncthreads();
        }
        if (!real) continue;
        const float tt = __fdiv_rn(bf16mag_to_f32(rmax), kNvfp4ScaleDivisor);
        const float six_t = __fmul_rn(6.0f, tt), four_t = __fmul_rn(4.0f, tt);
        // lane j < topk holds the slot of pair (t, j) (-1: not routed), and
        // that slot row's byte offsets: codes, and the row part of the
        // swizzled SF address (the block's column part is fixed per lane)
        const int32_t my_slot = lane < topk ? __ldg(slot_of + t * topk + lane) : -1;
        if (my_slot >= 0 && part == 0) scale[my_slot] = tt;
        const int64_t my_crow = (int64_t)(my_slot < 0 ? 0 : my_slot) * (H >> 1);
        const int64_t my_srow = my_slot < 0 ? 0 : sf_swizzled(my_slot, 0, ncol_tiles);
        uint2 cw[BPL];
        uint32_t sw[BPL];
#pragma unroll
        for (int i = 0; i < BPL; ++i) {
            const int b = li + 32 * WPR * i;
            uint2 c = make_uint2(0u, 0u);
            uint32_t s = 0;
            if (b < nblk && tt != 0.0f) {
                float xs[16];
                const uint32_t w[8] = {va[i].x, va[i].y, va[i].z, va[i].w, vb[i].x, vb[i].y, vb[i].z, vb[i].w};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    xs[2 * j] = bf16_lo(w[j]);
                    xs[2 * j + 1] = bf16_hi(w[j]);
                }
                const float ab = bf16mag_to_f32(bmax[i]);
                const BlockScale s6 = nvfp4_block_scale(ab, six_t, tt);
                c = encode16(xs, s6.enc);
                s = s6.sf;
                if (FOUR_SIX) {
                    const BlockScale s4 = nvfp4_block_scale(ab, four_t, tt);
                    const uint2 c4 = encode16(xs, s4.enc);
                    if (block_sse(xs, c4.x, c4.y, s4.d) < block_sse(xs, c.x, c.y, s6.d)) {
                        c = c4;
                        s = s4.sf;
                    }
                }
            }
            // the 4 scale bytes of blocks b .. b+3 (lanes b .. b+3) as one word:
            // consecutive in the swizzled layout, b % 4 == 0 at the gathering lane
            const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, s, 1);
            const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, s, 2);
            const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, s, 3);
            cw[i] = c;
            sw[i] = s | (s1 << 8) | (s2 << 16) | (s3 << 24);
        }
        // each routed slot: its code row, and the column part (b / 4) * 512 +
        // b % 4 of each block's swizzled SF address (b % 4 == 0 at the storing
        // lanes)
        for (int j = 0; j < topk; ++j) {
            const int32_t r = __shfl_sync(0xFFFFFFFFu, my_slot, j);
            if (r < 0) continue;  // warp-uniform
            const int64_t crow = __shfl_sync(0xFFFFFFFFu, my_crow, j);
            const int64_t srow = __shfl_sync(0xFFFFFFFFu, my_srow, j);
            uint2* cdst = reinterpret_cast<uint2*>(codes + crow);
            uint8_t* sdst = sf + srow;
#pragma unroll
            for (int i = 0; i < BPL; ++i) {
                const int b = li + 32 * WPR * i;
                if (b >= nblk) continue;
                cdst[b] = cw[i];
                if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(sdst + (b >> 2) * 512) = sw[i];
            }
        }
    }
}

// Combine: y[t] = sum_j w[t][j] * out[slot_of[t*k + j]], binary32 in
// ascending j, rounded to bf16.  One warp per token, 8 columns per lane step.
__global__ void __launch_bounds__(256) k_combine(const uint16_t* __restrict__ out, int64_t T, int64_t H,
                                                 int32_t topk, const int32_t* __restrict__ slot_of,
                                                 const float* __restrict__ w, uint16_t* __restrict__ y)
{
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
        // lane j < topk holds pair (t, j)'s slot and weight; broadcast below so
        // that a lane issues the loads of all k expert rows back to back
        const int32_t my_slot = lane < topk ? __ldg(slot_of + t * topk + lane) : -1;
        const float my_w = lane < topk ? __ldg(w + t * topk + lane) : 0.0f;
        for (int64_t c = 8 * lane; c < H; c += 256) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int j0 = 0; j0 < topk; j0 += 8) {
                uint4 v[8];
                float wj[8];
                bool has[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int j = j0 + jj;
                    const int32_t s = __shfl_sync(0xFFFFFFFFu, my_slot, j & 31);
                    wj[jj] = __shfl_sync(0xFFFFFFFFu, my_w, j & 31);
                    has[jj] = j < topk && s >= 0;
                    v[jj] = has[jj] ? __ldg(reinterpret_cast<const uint4*>(out + (int64_t)s * H + c))
                                    : make_uint4(0u, 0u, 0u, 0u);
                }
                // fixed order j = 0, 1, ...; pairs without a slot are skipped
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    if (!has[jj]) continue;
                    const uint32_t q[4] = {v[jj].x, v[jj].y, v[jj].z, v[jj].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(wj[jj], bf16_lo(q[i])));
                        acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(wj[jj], bf16_hi(q[i])));
                    }
                }
            }
            uint4 o;
            uint32_t* op = &o.x;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                op[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i])) |
                        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i + 1])) << 16);
            *reinterpret_cast<uint4*>(y + t * H + c) = o;
        }
    }
}

// ---------------------------------------------------------------------------
template <typename... KArgs, typename... Args>
static void launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args)
{
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

void launch_route(const int32_t* ids, int64_t T, int32_t topk, int32_t E, int32_t* hist, int32_t* counts,
                  int32_t* offsets, int32_t* slot_of, int32_t* row_src, int64_t capacity, int32_t* dev_status,
                  cudaStream_t st)
{
    const int64_t n = T * topk;
    const int nchunks = (int)((n + RT_CHUNK - 1) / RT_CHUNK);
    int32_t* ticket = hist + (int64_t)std::max(nchunks, 1) * E;  // one word after the histograms
    (void)capacity;  // row_src of padding rows and unused capacity: k_quant_scatter
    // the three phases with programmatic dependent launch: each starts while
    // the previous one drains and waits for it (pdl_enter) before its loads
    if (nchunks > 0) {
        launch_pdl(k_route_hist, dim3(nchunks), dim3(256), (size_t)E * sizeof(int32_t), st, ids, n, E, hist, ticket,
                   dev_status);
    } else {
        cudaMemsetAsync(ticket, 0, sizeof(int32_t), st);
    }
    launch_pdl(k_route_scan, dim3(E), dim3(256), 0, st, hist, nchunks, E, counts, offsets, ticket);
    if (nchunks > 0 && E <= RT_CTA_MAX_E)
        launch_pdl(k_route_assign_cta, dim3(nchunks), dim3(256), 0, st, ids, n, E, (const int32_t*)hist,
                   (const int32_t*)offsets, slot_of, row_src);
    else if (nchunks > 0)
        launch_pdl(k_route_assign, dim3(nchunks), dim3(32), (size_t)E * sizeof(int32_t), st, ids, n, E,
                   (const int32_t*)hist, (const int32_t*)offsets, slot_of, row_src);
}

void launch_quant_scatter(const uint16_t* x, int64_t T, int64_t H, int32_t topk, const int32_t* slot_of,
                          const int32_t* offsets, const int32_t* counts, int32_t E, uint8_t* codes, uint8_t* sf,
                          float* scale, int32_t* row_src, int64_t cap, bool four_six, int sms, cudaStream_t st)
{
    const int nblk = (int)(H >> 4);
    // one warp per token in CTAs of 4 warps: at ~70 registers a thread, an SM
    // holds 7 such CTAs (28 warps) against 3 CTAs of 8 warps (24)
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((T + 3) / 4, (int64_t)sms * 32));
#define BSQ_QS(B)                                                                                                  \
    do {                                                                                                           \
        if (four_six)                                                                                              \
            launch_pdl(k_quant_scatter<B, true>, dim3(grid), dim3(128), 0, st, x, T, H, topk, slot_of, offsets, counts, E, codes, sf, scale, row_src, cap); \
        else                                                                                                       \
            launch_pdl(k_quant_scatter<B, false>, dim3(grid), dim3(128), 0, st, x, T, H, topk, slot_of, offsets, counts, E, codes, sf, scale, row_src, cap); \
    } while (0)
    if (nblk <= 32) BSQ_QS(1);
    else if (nblk <= 64) BSQ_QS(2);
    else if (nblk <= 128) BSQ_QS(4);
    else {  // wide rows: 4 warps per token, up to 4 blocks per lane (H <= 8192)
        const int grid4 = (int)std::max<int64_t>(1, std::min<int64_t>((T + 1) / 2, (int64_t)sms * 16));
        if (four_six) launch_pdl(k_quant_scatter<4, true, 4>, dim3(grid4), dim3(256), 0, st, x, T, H, topk, slot_of, offsets, counts, E, codes, sf, scale, row_src, cap);
        else launch_pdl(k_quant_scatter<4, false, 4>, dim3(grid4), dim3(256), 0, st, x, T, H, topk, slot_of, offsets, counts, E, codes, sf, scale, row_src, cap);
    }
#undef BSQ_QS
}

void launch_combine(const uint16_t* out, int64_t T, int64_t H, int32_t topk, const int32_t* slot_of, const float* w,
                    uint16_t* y, int sms, cudaStream_t st)
{
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((T + 7) / 8, (int64_t)sms * 16));
    launch_pdl(k_combine, dim3(grid), dim3(256), 0, st, out, T, H, topk, slot_of, w, y);
}

}  // namespace bsq
