// gemm_fp4.cu -- NVFP4 x NVFP4 block-scaled grouped expert GEMM on the
// 5th-generation tensor cores (tcgen05.mma kind::mxf4nvf4, one E4M3 scale per
// 16 elements along K, fp32 accumulation in tensor memory), with the FP32
// per-token x per-expert rescale and the SwiGLU activation fused into the
// epilogue.
//
// Sources: block scales are applied by the tensor cores ("LMSYS Drops Miles
// ...", section "Why Blackwell changes the math"); the per-token FP32 scale
// belongs in the GEMM epilogue rather than in a separate pass (same page,
// section "Results"); SwiGLU experts run gate and up as one fused matmul
// ("Miles Blackwell RL ...", section "Un quantizzatore condiviso è il vero
// meccanismo").
//
// CTA = one 128-row x 256-column output tile of one expert (the grouped
// problem is flattened: 128-row tiles of the expert-sorted A, each inside one
// expert's segment, times the N tiles).  Warp roles (192 threads):
//   warp 0      TMA producer: A tile (128 x 256 fp4), B tile (2 x 128 rows),
//               and the SF chunks (512-byte tensor-core tiles) per stage
//   warp 1      allocates tensor memory; one lane copies SF into tensor memory
//               (tcgen05.cp) and issues the MMAs (128 x 128 x 64 each)
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (warp w reads lanes
//               32*(w%4)..+31), rescale, SwiGLU, stores
// Shared memory: GM_STAGES stages of [SFA 2 KB][SFB 4 KB][A 16 KB][B 32 KB]
// (A and B 128-byte swizzled, 1024-byte aligned).  Tensor memory: 512 columns
// = accumulator (256) + an SF ring (48 per stage).
// Every mbarrier wait is bounded; on expiry the CTA records BSQ_DEV_TIMEOUT,
// drains its outstanding copies and MMAs (bounded), frees tensor memory and
// returns.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace bsq {

constexpr int GM_THREADS = 192;
constexpr int GM_STAGES = 4;
constexpr int GM_SFA_OFF = 0;
constexpr int GM_SFB_OFF = 2048;
constexpr int GM_A_OFF = 6144;
constexpr int GM_B_OFF = 6144 + 16384;
constexpr int GM_STAGE_BYTES = 6144 + 16384 + 32768;  // 55296 = 54 KB
constexpr int GM_TMEM_COLS = 512;
constexpr int GM_SF_RING = 256;                       // first SF column
constexpr int GM_SF_STAGE_COLS = 48;
constexpr uint32_t GM_SPIN_LIMIT = 1u << 22;
constexpr size_t GM_SMEM_BYTES = (size_t)GM_STAGES * GM_STAGE_BYTES + 1024 + 1024;

// Instruction descriptor, kind::mxf4nvf4: A and B are E2M1 (format 1),
// K-major, no negation, N = 128 (N>>3 at bit 17), M = 128 (M>>4 at bit 24),
// scale type UE4M3 (bit 23 = 0), scale-factor ids 0, dense.
constexpr uint32_t GM_IDESC = (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

// ------------------------------------------------------------------ PTX
BSQ_DEVICE uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

BSQ_DEVICE void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
BSQ_DEVICE void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
BSQ_DEVICE bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait; gives up when the abort flag is raised or the spin limit hit.
BSQ_DEVICE bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag)
{
    for (uint32_t i = 0; i < GM_SPIN_LIMIT; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && *abort_flag) return false;
    }
    return false;
}

BSQ_DEVICE void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
BSQ_DEVICE void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

BSQ_DEVICE void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
BSQ_DEVICE void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
BSQ_DEVICE void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Shared-memory matrix descriptor: start >> 4 (bits 0-13), leading byte
// offset >> 4 (16-29), stride byte offset >> 4 (32-45), version 1 (46),
// swizzle mode (61-63: 0 none, 2 = 128-byte).
BSQ_DEVICE uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)swz << 61);
}

BSQ_DEVICE void tc_cp_sf(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

BSQ_DEVICE void tc_mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                       uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
}

BSQ_DEVICE void tc_ld32(uint32_t taddr, float v[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

BSQ_DEVICE uint32_t pack_bf16x2(float lo, float hi)
{
    const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return l | (h << 16);
}

BSQ_DEVICE float silu(float g) { return g / (1.0f + __expf(-g)); }

// ------------------------------------------------------------------ kernel
struct GemmParams {
    const uint8_t* a_sf;
    const float* a_scale;
    const int32_t* offsets;
    const uint8_t* b_sf;
    const float* b_scale;
    void* out;
    int32_t* dev_status;
    int64_t ldo;
    int32_t experts;
    int32_t m_capacity;
    int32_t K;
    int32_t N;
    int32_t n_tiles;
    int32_t epilogue;
};

__global__ void __launch_bounds__(GM_THREADS, 1)
    k_gemm_fp4(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[2 * GM_STAGES + 2];
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nt = blockIdx.x % p.n_tiles;
    const int m0 = (blockIdx.x / p.n_tiles) * 128;

    // ---- which expert owns rows [m0, m0+128)?
    const int E = p.experts;
    const int total = __ldg(p.offsets + E);
    if (m0 >= total) return;  // beyond the routed rows: nothing to do (no barrier/TMEM touched yet)
    int lo = 0, hi = E - 1;   // largest e with offsets[e] <= m0
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(p.offsets + mid) <= m0) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    {
        // segment starts are multiples of 128; the total (offsets[E]) need not be
        const int seg0 = __ldg(p.offsets + e), seg1 = __ldg(p.offsets + e + 1);
        if ((seg0 & 127) || (e + 1 < E && (seg1 & 127)) || seg1 < seg0 || total > p.m_capacity || total < 0) {
            if (threadIdx.x == 0) report(p.dev_status, BSQ_DEV_BAD_OFFSETS);
            return;
        }
    }

    const bool swiglu = p.epilogue == BSQ_EPI_SWIGLU_BF16;
    const int n_halves = swiglu ? 2 : ((nt * 256 + 128 < p.N) ? 2 : 1);
    const int brow0 = swiglu ? e * p.N + nt * 128 : e * p.N + nt * 256;
    const int brow1 = swiglu ? e * p.N + (p.N >> 1) + nt * 128 : brow0 + 128;
    const int k64_total = p.K >> 6;
    const int kt_count = (k64_total + 3) >> 2;

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(GM_STAGES + s); };
    const uint32_t acc_bar = bar0 + 8u * (2 * GM_STAGES);
    const uint32_t drain_bar = bar0 + 8u * (2 * GM_STAGES + 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < GM_STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(acc_bar, 1);
        mbar_init(drain_bar, 1);
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem_base)),
                     "r"(GM_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem_base;
    volatile int* abort_flag = &s_abort;

    if (warp == 0) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
            const uint8_t* sfa_src = p.a_sf + ((size_t)(m0 >> 7) * k64_total) * 512;
            const uint8_t* sfb_src0 = p.b_sf + ((size_t)(brow0 >> 7) * k64_total) * 512;
            const uint8_t* sfb_src1 = p.b_sf + ((size_t)(brow1 >> 7) * k64_total) * 512;
            int issued = 0;
            for (int kt = 0; kt < kt_count; ++kt) {
                const int s = kt % GM_STAGES;
                const uint32_t ph = (uint32_t)(kt / GM_STAGES) & 1u;
                if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag)) {
                    *abort_flag = 1;
                    report(p.dev_status, BSQ_DEV_TIMEOUT);
                    break;
                }
                const int nk = min(4, k64_total - 4 * kt);
                const uint32_t sf_bytes = (uint32_t)nk * 512u;
                const uint32_t bytes = 16384u + 16384u * (uint32_t)n_halves + sf_bytes * (uint32_t)(1 + n_halves);
                const uint32_t st = sbase + (uint32_t)s * GM_STAGE_BYTES;
                mbar_expect_tx(full_bar(s), bytes);
                tma_load_2d(st + GM_A_OFF, &tmA, kt * 128, m0, full_bar(s));
                tma_load_2d(st + GM_B_OFF, &tmB, kt * 128, brow0, full_bar(s));
                if (n_halves == 2) tma_load_2d(st + GM_B_OFF + 16384, &tmB, kt * 128, brow1, full_bar(s));
                bulk_load(st + GM_SFA_OFF, sfa_src + (size_t)kt * 2048, sf_bytes, full_bar(s));
                bulk_load(st + GM_SFB_OFF, sfb_src0 + (size_t)kt * 2048, sf_bytes, full_bar(s));
                if (n_halves == 2) bulk_load(st + GM_SFB_OFF + 2048, sfb_src1 + (size_t)kt * 2048, sf_bytes, full_bar(s));
                ++issued;
            }
            if (*abort_flag) {
                // let the copies already issued land before the CTA exits
                for (int kt = max(0, issued - GM_STAGES); kt < issued; ++kt) {
                    for (uint32_t i = 0; i < GM_SPIN_LIMIT; ++i)
                        if (mbar_try_wait(full_bar(kt % GM_STAGES), (uint32_t)(kt / GM_STAGES) & 1u)) break;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool issued_any = false;
            for (int kt = 0; kt < kt_count; ++kt) {
                const int s = kt % GM_STAGES;
                const uint32_t ph = (uint32_t)(kt / GM_STAGES) & 1u;
                if (!mbar_wait(full_bar(s), ph, abort_flag)) {
                    *abort_flag = 1;
                    report(p.dev_status, BSQ_DEV_TIMEOUT);
                    break;
                }
                tc_fence_after();
                const int nk = min(4, k64_total - 4 * kt);
                const uint32_t st = sbase + (uint32_t)s * GM_STAGE_BYTES;
                const uint32_t sf_col = tmem + GM_SF_RING + (uint32_t)s * GM_SF_STAGE_COLS;
                for (int j = 0; j < nk; ++j) {
                    tc_cp_sf(sf_col + 4 * j, smem_desc(st + GM_SFA_OFF + 512 * j, 16, 128, 0));
                    tc_cp_sf(sf_col + 16 + 4 * j, smem_desc(st + GM_SFB_OFF + 512 * j, 16, 128, 0));
                    if (n_halves == 2)
                        tc_cp_sf(sf_col + 32 + 4 * j, smem_desc(st + GM_SFB_OFF + 2048 + 512 * j, 16, 128, 0));
                }
                for (int j = 0; j < nk; ++j) {
                    const uint64_t ad = smem_desc(st + GM_A_OFF + 32 * j, 16, 1024, 2);
                    const uint32_t acc = (kt > 0 || j > 0) ? 1u : 0u;
                    for (int h = 0; h < n_halves; ++h) {
                        const uint64_t bd = smem_desc(st + GM_B_OFF + 16384 * h + 32 * j, 16, 1024, 2);
                        tc_mma(tmem + 128 * h, ad, bd, GM_IDESC, sf_col + 4 * j, sf_col + 16 + 16 * h + 4 * j, acc);
                    }
                }
                tc_commit(empty_bar(s));
                issued_any = true;
            }
            if (!*abort_flag) {
                tc_commit(acc_bar);
                // tensor memory is freed only after the last MMA has completed
                for (uint32_t i = 0; i < GM_SPIN_LIMIT; ++i)
                    if (mbar_try_wait(acc_bar, 0u)) break;
            } else if (issued_any) {
                tc_commit(drain_bar);  // completes when every MMA/copy issued so far has finished
                for (uint32_t i = 0; i < GM_SPIN_LIMIT; ++i)
                    if (mbar_try_wait(drain_bar, 0u)) break;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int row = m0 + 32 * q + lane;
        const bool ok = mbar_wait(acc_bar, 0u, abort_flag);
        if (__all_sync(0xFFFFFFFFu, ok)) {
            tc_fence_after();
            const bool in = row < p.m_capacity;
            const float s = in ? __fmul_rn(__ldg(p.a_scale + row), __ldg(p.b_scale + e)) : 0.0f;
            const uint32_t tlane = tmem + ((uint32_t)(32 * q) << 16);
            if (swiglu) {
                const int I = p.N >> 1;
                __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + (size_t)row * p.ldo + nt * 128;
                for (int c = 0; c < 4; ++c) {
                    float g[32], u[32];
                    tc_ld32(tlane + 32 * c, g);
                    tc_ld32(tlane + 128 + 32 * c, u);
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float h0 = silu(__fmul_rn(g[2 * i], s)) * __fmul_rn(u[2 * i], s);
                        const float h1 = silu(__fmul_rn(g[2 * i + 1], s)) * __fmul_rn(u[2 * i + 1], s);
                        w[i] = pack_bf16x2(h0, h1);
                    }
                    if (in && nt * 128 + 32 * c < I) {
                        uint4* d = reinterpret_cast<uint4*>(o + 32 * c);
#pragma unroll
                        for (int i = 0; i < 4; ++i) d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    }
                }
            } else {
                const int n0 = nt * 256;
                for (int c = 0; c < 4 * n_halves; ++c) {
                    float v[32];
                    tc_ld32(tlane + 32 * c, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(v[i], s);
                    if (!in) continue;
                    if (p.epilogue == BSQ_EPI_F32) {
                        float4* d = reinterpret_cast<float4*>(static_cast<float*>(p.out) + (size_t)row * p.ldo + n0 + 32 * c);
#pragma unroll
                        for (int i = 0; i < 8; ++i) d[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    } else {
                        uint4* d = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + (size_t)row * p.ldo + n0 + 32 * c);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            d[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                              pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
                    }
                }
            }
        } else if (lane == 0) {
            *abort_flag = 1;
            report(p.dev_status, BSQ_DEV_TIMEOUT);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(GM_TMEM_COLS) : "memory");
    }
}

// ------------------------------------------------------------------ host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D byte tensor [rows][row_bytes], box 128 x 128 bytes, 128-byte swizzle.
static bool make_tmap(CUtensorMap* tm, const void* base, int64_t rows, int64_t row_bytes)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {128u, 128u};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_gemm_fp4(const GemmArgs& a, cudaStream_t st)
{
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t err = cudaFuncSetAttribute(k_gemm_fp4, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)GM_SMEM_BYTES);
        if (err != cudaSuccess) return err;
        attr_set = true;
    }
    CUtensorMap tmA, tmB;
    if (!make_tmap(&tmA, a.a_codes, a.m_capacity, a.K / 2)) return cudaErrorInvalidValue;
    if (!make_tmap(&tmB, a.b_codes, a.experts * a.N, a.K / 2)) return cudaErrorInvalidValue;
    GemmParams p;
    p.a_sf = a.a_sf;
    p.a_scale = a.a_scale;
    p.offsets = a.offsets;
    p.b_sf = a.b_sf;
    p.b_scale = a.b_scale;
    p.out = a.out;
    p.dev_status = a.dev_status;
    p.ldo = a.ldo;
    p.experts = (int32_t)a.experts;
    p.m_capacity = (int32_t)a.m_capacity;
    p.K = (int32_t)a.K;
    p.N = (int32_t)a.N;
    p.epilogue = a.epilogue;
    p.n_tiles = a.epilogue == BSQ_EPI_SWIGLU_BF16 ? (int32_t)(a.N / 256) : (int32_t)((a.N + 255) / 256);
    const int64_t m_tiles = (a.m_capacity + 127) / 128;
    const int64_t grid = m_tiles * p.n_tiles;
    if (grid == 0) return cudaSuccess;
    k_gemm_fp4<<<(unsigned)grid, GM_THREADS, GM_SMEM_BYTES, st>>>(tmA, tmB, p);
    return cudaGetLastError();
}

}  // namespace bsq
