// gemm_fp4.cu -- NVFP4 x NVFP4 block-scaled grouped expert GEMM on the
// 5th-generation tensor cores (tcgen05.mma kind::mxf4nvf4, one E4M3 scale per
// 16 elements along K, fp32 accumulation in tensor memory), with the FP32
// per-token x per-expert rescale and the SwiGLU activation fused into the
// epilogue; the same pipeline runs MXFP8 operands (kind::mxf8f6f4).
//
// Sources: block scales are applied by the tensor cores ("LMSYS Drops Miles
// ...", section "Why Blackwell changes the math"); the per-token FP32 scale
// belongs in the GEMM epilogue rather than in a separate pass (same page,
// section "Results"); SwiGLU experts run gate and up as one fused matmul
// ("Miles Blackwell RL ...", section "Un quantizzatore condiviso è il vero
// meccanismo"); on GB300 the FP4 tensor cores are fast enough that feeding
// them is the hard part, which a 2-SM MMA addresses ("End-to-End 4-Bit
// Training", section "工程细节").
//
// Persistent kernel, one CTA per SM, in one of two forms (CG):
//   CG = 2  clusters of two CTAs on neighbouring SMs share each MMA
//           (tcgen05.mma.cta_group::2, 256 x 256 x 64): the pair computes a
//           256-row x 256-column output tile, each CTA holding 128 rows of A
//           and 128 of B's 256 N rows in its shared memory and receiving its
//           128 rows of D in its tensor memory.  B is read from shared memory
//           once for both SMs, so a 256-wide K stage costs each SM 38 KB of
//           copies and 32 KB of operand reads instead of 54 KB and 48 KB:
//           the per-SM shared-memory traffic, not the MMA rate, is what
//           bounds this GEMM.  A pair tile lies inside one expert's segment
//           (segments are padded to 128 rows, so an odd count of 128-row
//           tiles leaves a last pair tile whose second half is not stored).
//   CG = 1  one CTA per 128 x 256 tile (for more experts than the pair
//           schedule keeps in shared memory).
// Tiles are walked round-robin by CTA (CG 1) or pair (CG 2), N fastest.
//   warp 0      TMA producer, in every CTA.  Per stage it first copies the
//               scale factors (SFA: 2 KB for its 128 rows; SFB: the 4 KB of
//               all 256 N rows, which every CTA's tensor memory needs) on the
//               scale-factor barrier, then the codes: A (128 x 128 B) and B
//               (256 rows with CG 1; its 128-row half with CG 2).  With CG 2
//               both CTAs' copies complete on the first CTA's barriers.
//   warp 1      allocates tensor memory; in the first CTA one lane issues the
//               MMAs (four per stage) and the commits, which with CG 2 reach
//               the barriers of both CTAs
//   warps 2..   one or three scale-factor movers (first CTA): as soon as a
//               stage's scale factors land, tcgen05.cp 32x128b.warpx4 moves
//               them into tensor memory (with CG 2, each CTA's chunk into its
//               own) while the codes are still in flight
//   the last 16 warps  epilogue, in every CTA, four per lane quadrant, 64
//               columns each: load the accumulator, hand it back to the MMA
//               warp, then rescale / SwiGLU / store while the next tile's MMAs
//               run
// Shared memory: a ring of stages of [SFA 2 KB][SFB 4 KB][A 16 KB][B 16/32 KB]
// (A and B 128-byte swizzled, 1024-byte aligned) and the expert offsets; the
// plain bf16 epilogue adds a 2 KB staging buffer per epilogue warp (one TMA
// tensor store per 32 x 32 block).  The ring's depth hides the round trip of
// a stage (MMAs complete -> stage released -> copies issued -> copies landed).
// Tensor memory: 512 columns = accumulator (256) + an SF ring (48 per stage:
// SFA k-step j at 4j, SFB k-step j at 16 + 8j, both N halves side by side).
// Every mbarrier wait is bounded; on expiry the CTA records BSQ_DEV_TIMEOUT,
// stops issuing, lets its outstanding copies and MMAs finish (bounded), frees
// tensor memory and returns.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace bsq {

constexpr int GM_MAX_SF_WARPS = 3;
constexpr int GM_EPI_WARPS = 16;
constexpr int GM_MAX_STAGES = 5;
constexpr int GM_SFA_OFF = 0;
constexpr int GM_SFB_OFF = 2048;
constexpr int GM_A_OFF = 6144;
constexpr int GM_B_OFF = 6144 + 16384;
constexpr int GM_TMEM_COLS = 512;
constexpr int GM_SF_RING = 256;                       // first SF column
constexpr int GM_SF_STAGE_COLS = 48;
constexpr int GM_MAX_SMEM_EXPERTS = 256;              // offsets cached in shared memory up to this E
#ifdef BSQ_GEMM_STALL_HOOK
// Test build only (never the product library): the producer issues no copies
// and never arrives, and every wait gives up after a few thousand polls, so
// each role takes its timeout path with nothing asynchronous in flight.
constexpr uint32_t GM_SPIN_LIMIT = 1u << 12;
constexpr bool GM_STALL = true;
#else
constexpr uint32_t GM_SPIN_LIMIT = 1u << 22;
constexpr bool GM_STALL = false;
#endif
constexpr int GM_EPI_WARP_BYTES = 32 * 64;            // 32 rows x 64 bytes, 64-byte swizzled

// Per epilogue kind and form: the stage count, whether the epilogue stages its
// stores through shared memory (after the ring), the dynamic shared memory,
// and the number of scale-factor mover warps.  Two movers (six of a stage's
// twelve chunk copies each) get the scale factors into tensor memory soonest,
// which the long-K SwiGLU GEMM needs; at 20 warps (five per SM sub-partition)
// a thread keeps 96 registers, which the SwiGLU epilogue needs to run without
// spills.  One mover keeps the bf16 GEMM at 19 warps.  The pair form's 38 KB
// stages fit five deep.
template <int EPI>
constexpr bool gm_swiglu = EPI == BSQ_EPI_SWIGLU_BF16 || EPI == GM_EPI_SWIGLU_Q || EPI == GM_EPI_SWIGLU_Q46;
template <int EPI>
constexpr bool gm_fused_q = EPI == GM_EPI_SWIGLU_Q || EPI == GM_EPI_SWIGLU_Q46;

template <int EPI, int CG>
struct GmCfg {
    static constexpr int SF_WARPS = gm_swiglu<EPI> ? 2 : 1;
    static constexpr int THREADS = 32 * (2 + SF_WARPS + GM_EPI_WARPS);
    static constexpr bool STAGED = EPI == BSQ_EPI_BF16;
    static constexpr int B_BYTES = CG == 2 ? 16384 : 32768;
    static constexpr int STAGE_BYTES = GM_B_OFF + B_BYTES;  // 38 KB / 54 KB
    static constexpr int STAGES = CG == 2 ? 5 : (STAGED ? 3 : 4);
    static constexpr int EPI_OFF = STAGES * STAGE_BYTES;
    static constexpr size_t SMEM_BYTES =
        (size_t)EPI_OFF + (STAGED ? (size_t)GM_EPI_WARPS * GM_EPI_WARP_BYTES : 0) + 1024;
};
static_assert(GM_SF_RING + GM_MAX_STAGES * GM_SF_STAGE_COLS <= GM_TMEM_COLS, "SF ring exceeds tensor memory");
static_assert(GmCfg<BSQ_EPI_BF16, 2>::SMEM_BYTES + 2560 <= 232448, "stage ring exceeds shared memory");
static_assert(GmCfg<BSQ_EPI_SWIGLU_BF16, 1>::SMEM_BYTES + 3584 <= 232448, "stage ring exceeds shared memory");
static_assert(GmCfg<GM_EPI_SWIGLU_Q, 2>::SMEM_BYTES + 3584 <= 232448, "stage ring exceeds shared memory");

// Bounded wait; gives up when the abort flag is raised or the spin limit hit.
// CLUSTER: acquire at cluster scope, for a barrier the other CTA of a pair
// arrives on.
template <bool CLUSTER = false>
BSQ_DEVICE bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag)
{
    for (uint32_t i = 0; i < GM_SPIN_LIMIT; ++i) {
        if (CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && *abort_flag) return false;
    }
    return false;
}
// The same by a whole converged warp: every lane polls, and the lanes agree
// on the outcome (the producer, MMA and scale-factor roles run warp-wide so
// that their tcgen05 and TMA operands stay warp-uniform).
template <bool CLUSTER = false>
BSQ_DEVICE bool mbar_wait_w(uint32_t bar, uint32_t parity, volatile int* abort_flag)
{
    for (uint32_t i = 0; i < GM_SPIN_LIMIT; ++i) {
        const bool done = CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
        if (__all_sync(0xFFFFFFFFu, done)) return true;
        if ((i & 255u) == 255u && __any_sync(0xFFFFFFFFu, *abort_flag != 0)) return false;
    }
    return false;
}
BSQ_DEVICE bool aborted_w(volatile int* abort_flag) { return __any_sync(0xFFFFFFFFu, *abort_flag != 0); }
// Bounded wait that ignores the abort flag (the drains before tensor memory
// is freed).
BSQ_DEVICE void mbar_drain(uint32_t bar, uint32_t parity)
{
    for (uint32_t i = 0; i < GM_SPIN_LIMIT; ++i)
        if (mbar_try_wait(bar, parity)) return;
}

BSQ_DEVICE uint32_t pack_bf16x2(float lo, float hi)
{
    const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return l | (h << 16);
}


// h = silu(g) * u = g * u / (1 + e^-g).  The exponential is the hardware
// approximation (__expf); the reciprocal r of d = 1 + e^-g uses the FMA pipe
// instead of a second special-function operation (the SwiGLU epilogue is
// bound by those): an estimate from d's IEEE-754 bit pattern (its exponent
// negated by subtracting the bits from a constant, 0x7EF311C2, found by a
// minimax search over one binade: relative error <= 5.1%), then two
// Newton-Raphson steps r <- r (2 - d r), which square the relative error:
// <= 7e-6, far below the bf16 rounding of h.  d is clamped to 1e30 so that
// e^-g = inf gives h -> 0, the limit.
BSQ_DEVICE float swiglu1(float g, float u)
{
    const float d = fminf(1.0f + __expf(-g), 1e30f);
    float r = __uint_as_float(0x7EF311C2u - __float_as_uint(d));
    r = r * (2.0f - d * r);
    r = r * (2.0f - d * r);
    return g * u * r;
}

// The epilogue's bf16 block store: thread `lane` owns row `lane` of a 32 x 32
// bf16 block (64 bytes).  The warp's buffer uses the TMA 64-byte swizzle
// (16-byte chunk c of row r lives at chunk c ^ ((r >> 1) & 3)), which also
// keeps the 16-byte writes of each quarter-warp on distinct banks; one lane
// then stores the block with a TMA tensor store (rows past the tensor map's
// extent are clipped by the hardware).
BSQ_DEVICE void stage_put(uint8_t* buf, int lane, int c, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3)
{
    *reinterpret_cast<uint4*>(buf + 64 * lane + 16 * (c ^ ((lane >> 1) & 3))) = make_uint4(w0, w1, w2, w3);
}
BSQ_DEVICE void stage_store(const uint8_t* buf, int lane, const CUtensorMap* tm, int x, int y)
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
        asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                         reinterpret_cast<uint64_t>(tm)),
                     "r"(x), "r"(y), "r"(smem_u32(buf))
                     : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
}
// The buffer may be rewritten once the previous store has read it.
BSQ_DEVICE void stage_reuse(int lane)
{
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    __syncwarp();
}

// 32 bytes of one output row straight from registers: one 256-bit store (a
// whole 32-byte sector per lane) when the destination is 32-byte aligned, else
// two 128-bit stores.
BSQ_DEVICE void st_row32(void* ptr, const uint32_t* w, bool vec32)
{
    if (vec32) {
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                     : "memory");
    } else {
        uint4* q = static_cast<uint4*>(ptr);
        q[0] = make_uint4(w[0], w[1], w[2], w[3]);
        q[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

// The per-token NVFP4 quantization of 128 rows of h (a GEMM1 unit) whose row
// maxima, as bf16 magnitude bits, are already in smax (each is reset to 0 once
// read): half-warp hw of 32 takes rows hw, hw + 32, ...; lane lr of it blocks
// lr, lr + 16, ..., two at a time with their loads issued first.  The same
// arithmetic as the per-token quantizer (nvfp4_block).
template <bool FOUR_SIX>
BSQ_DEVICE void gm_quantize_h_rows(uint32_t* smax, const uint8_t* hb, int64_t ldo, int nblk, int r0,
                                                int m_capacity, uint8_t* q_codes, uint8_t* q_sf, float* q_scale,
                                                int hw, int lr)
{
    for (int rr = hw; rr < 128; rr += 2 * GM_EPI_WARPS) {
        const int grow = r0 + rr;
        const uint32_t amax = smax[rr];
        __syncwarp();
        if (lr == 0) smax[rr] = 0u;  // the buffer's next unit comes after the next meeting
        if (grow >= m_capacity) continue;
        const float tq = __fdiv_rn(bf16mag_to_f32(amax), kNvfp4ScaleDivisor);
        const float six_t = __fmul_rn(6.0f, tq), four_t = __fmul_rn(4.0f, tq);
        const uint8_t* hr = hb + (size_t)rr * ldo * 2;
        uint2* crow = reinterpret_cast<uint2*>(q_codes + (size_t)grow * (nblk * 8));
        for (int b0 = lr; b0 < nblk; b0 += 32) {
            uint4 va[2], vb[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int b = b0 + 16 * i;
                if (b < nblk) {
                    va[i] = __ldcg(reinterpret_cast<const uint4*>(hr + 32 * b));
                    vb[i] = __ldcg(reinterpret_cast<const uint4*>(hr + 32 * b + 16));
                }
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int b = b0 + 16 * i;
                if (b < nblk) {
                    uint2 c;
                    uint32_t sfv;
                    nvfp4_block<FOUR_SIX>(va[i], vb[i], absmax16(va[i], vb[i]), tq, six_t, four_t, c, sfv);
                    crow[b] = c;
                    q_sf[sf_swizzled(grow, b, nblk >> 2)] = (uint8_t)sfv;
                }
            }
        }
        if (lr == 0) q_scale[grow] = tq;
    }
}

// ------------------------------------------------------------------ kernel
struct GemmParams {
    const uint8_t* a_sf;
    const uint8_t* b_sf;
    const float* a_scale;
    const int32_t* offsets;
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
    bool out_vec32;  // output base and row pitch are 32-byte aligned
    // fused quantization of h (GM_EPI_SWIGLU_Q*): NVFP4 h [m_capacity][N/4 bytes],
    // its swizzled SF and per-row scale; the per-CTA bf16 scratch (128 x N/2),
    // or h kept whole in `out` when keep_h
    uint8_t* q_codes;
    uint8_t* q_sf;
    float* q_scale;
    uint16_t* h_scratch;
    bool keep_h;
};

struct TileInfo {
    int m0, nt, e, n_halves, seg_end;
};

// EPI is the epilogue (BSQ_EPI_*): one instantiation per epilogue keeps each
// one's register allocation to its own path.  FMT is the operand format:
// 0 NVFP4 (E2M1 codes, E4M3 scale per 16, kind::mxf4nvf4, K = 64 per MMA,
// four 512-byte scale chunks per 128 rows and stage), 1 MXFP8 (E4M3 codes,
// E8M0 scale per 32, kind::mxf8f6f4, K = 32 per MMA, one chunk per 128 rows
// and stage).  A stage is 128 bytes of every row in both.  CG is the form
// (see the top of the file).
template <int EPI, int FMT, int CG>
__global__ void __launch_bounds__(GmCfg<EPI, CG>::THREADS, 1)
    k_gemm_fp4(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
               const __grid_constant__ CUtensorMap tmOut, const GemmParams p)
{
    using Cfg = GmCfg<EPI, CG>;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int SF_WARPS = Cfg::SF_WARPS;
    constexpr int STAGE_BYTES = Cfg::STAGE_BYTES;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[4 * GM_MAX_STAGES + 3 + GM_MAX_SF_WARPS];
    __shared__ int32_t s_off[GM_MAX_SMEM_EXPERTS + 1];
    __shared__ int32_t s_poff[CG == 2 ? GM_MAX_SMEM_EXPERTS + 1 : 1];  // first pair tile of each expert
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort, s_bad;
    // with the fused quantization of h: each row's running max |h| (bf16
    // magnitude bits) over a unit's N tiles, double-buffered by unit
    __shared__ uint32_t s_hmax[gm_fused_q<EPI> ? 2 : 1][128];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;  // the pair's first CTA issues the MMAs
    const int E = p.experts;
    const bool off_in_smem = E <= GM_MAX_SMEM_EXPERTS;  // always, with CG 2 (host checks)
    for (int i = threadIdx.x; i <= E && off_in_smem; i += blockDim.x) s_off[i] = __ldg(p.offsets + i);

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(STAGES + s); };
    auto sf_bar = [&](int s) { return bar0 + 8u * (uint32_t)(2 * STAGES + s); };
    auto sf_full = [&](int s) { return bar0 + 8u * (uint32_t)(3 * STAGES + s); };
    const uint32_t acc_full = bar0 + 8u * (4 * STAGES);
    const uint32_t acc_empty = bar0 + 8u * (4 * STAGES + 1);
    const uint32_t drain_bar = bar0 + 8u * (4 * STAGES + 2);
    auto sf_drain = [&](int w) { return bar0 + 8u * (uint32_t)(4 * STAGES + 3 + w); };
    // the first CTA's barrier at the same offset, as a shared::cluster address
    auto lead = [&](uint32_t bar) { return CG == 2 ? mapa_shared(bar, 0u) : bar; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);  // with CG 2 the first CTA expects both CTAs' bytes
            mbar_init(empty_bar(s), 1);
            mbar_init(sf_bar(s), SF_WARPS);
            mbar_init(sf_full(s), 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, CG * GM_EPI_WARPS);
        mbar_init(drain_bar, 32);  // every lane of the issuing warp commits (tc_commit_all)
        for (int w = 0; w < SF_WARPS; ++w) mbar_init(sf_drain(w), 32);
        s_abort = 0;
        for (int i = 0; i < (gm_fused_q<EPI> ? 256 : 128); ++i) (&s_hmax[0][0])[i] = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) tmem_alloc<CG>(smem_u32(&s_tmem_base), GM_TMEM_COLS);
    tc_fence_before();
    if constexpr (CG == 2)
        cluster_sync();  // the peer's barriers are initialised before any copy or arrival reaches them
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem_base;
    volatile int* abort_flag = &s_abort;

    auto off = [&](int i) { return off_in_smem ? s_off[i] : __ldg(p.offsets + i); };
    // Offsets contract: ascending, segment starts multiples of 128, total <= capacity.
    if (threadIdx.x == 0) {
        int bad = 0;
        for (int i = 0; i < E && !bad; ++i) {
            const int a = off(i), b = off(i + 1);
            bad = (a & 127) || b < a;
        }
        const int total = off(E);
        bad = bad || total > p.m_capacity || total < 0;
        s_bad = bad;
        if (bad && rank == 0) report(p.dev_status, BSQ_DEV_BAD_OFFSETS);
    }
    __syncthreads();
    if constexpr (CG == 2) {
        // pair tiles: expert e's ceil(tiles_e / 2) tiles of 256 rows, numbered
        // consecutively; warp 0 scans the counts, 8 experts per lane
        if (warp == 0 && !s_bad) {
            int cnt[8], sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = 8 * lane + j;
                cnt[j] = e < E ? ((((s_off[e + 1] - s_off[e]) + 127) >> 7) + 1) >> 1 : 0;
                sum += cnt[j];
            }
            int incl = sum;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if (lane >= d) incl += v;
            }
            int run = incl - sum;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int e = 8 * lane + j;
                if (e < E) s_poff[e] = run;
                run += cnt[j];
            }
            if (lane == 31) s_poff[E] = incl;
        }
        __syncthreads();
    }

    constexpr bool swiglu = gm_swiglu<EPI>;
    constexpr bool fused = gm_fused_q<EPI>;
    const int kmma_total = FMT ? (p.K >> 5) : (p.K >> 6);  // MMAs along K (64 or 32 elements each)
    const int kt_count = (kmma_total + 3) >> 2;
    const int sf_chunks = FMT ? (p.K >> 7) : (p.K >> 6);  // 512-byte scale chunks per 128-row tile
    const int m_units = s_bad ? 0 : (CG == 2 ? s_poff[E] : (off(E) + 127) >> 7);
    const int total_tiles = m_units * p.n_tiles;
    const int unit0 = (int)blockIdx.x / CG, unit_step = (int)gridDim.x / CG;
    // The k-th tile of this CTA (pair): round-robin over the tiles, or, with the
    // fused quantization of h, round-robin over the M units with each unit's N
    // tiles in order, so that all of a row's h is produced on this CTA
    auto tile_of = [&](int k) {
        if constexpr (fused) {
            const int u = unit0 + (k / p.n_tiles) * unit_step;
            return u < m_units ? u * p.n_tiles + k % p.n_tiles : total_tiles;
        } else {
            return unit0 + k * unit_step;
        }
    };

    auto tile_info = [&](int tile) {
        TileInfo t;
        t.nt = tile % p.n_tiles;
        const int mu = tile / p.n_tiles;
        int lo = 0, hi = E - 1;  // largest e whose first row (CG 1) / pair tile (CG 2) is <= the unit's
        if constexpr (CG == 2) {
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_poff[mid] <= mu) lo = mid; else hi = mid - 1;
            }
            t.m0 = off(lo) + 256 * (mu - s_poff[lo]);
        } else {
            t.m0 = mu * 128;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (off(mid) <= t.m0) lo = mid; else hi = mid - 1;
            }
        }
        t.e = lo;
        t.seg_end = off(lo + 1);
        t.n_halves = swiglu ? 2 : ((t.nt * 256 + 128 < p.N) ? 2 : 1);
        return t;
    };
    // with CG 2: whether this CTA's 128 rows of the pair tile are in the expert's segment
    auto half_valid = [&](const TileInfo& t) { return CG == 1 || rank == 0 || t.m0 + 128 < t.seg_end; };

    if (warp == 0) {
        // ------------------------------------------------------ producer (every CTA, whole warp)
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmSFB)) : "memory");
            if (CG == 2) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmSFA)) : "memory");
        }
        __syncwarp();
        uint32_t it = 0;
        for (int k = 0; !GM_STALL && !aborted_w(abort_flag); ++k) {
            const int tile = tile_of(k);
            if (tile >= total_tiles) break;
            const TileInfo t = tile_info(tile);
            const int my_m0 = t.m0 + 128 * (int)rank;  // this CTA's 128 rows of A
            const uint8_t* sfa_src = p.a_sf + ((size_t)(my_m0 >> 7) * sf_chunks) * 512;
            for (int kt = 0; kt < kt_count; ++kt, ++it) {
                const int s = (int)(it % STAGES);
                const uint32_t ph = (it / STAGES) & 1u;
                if (!mbar_wait_w(empty_bar(s), ph ^ 1u, abort_flag)) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        report(p.dev_status, BSQ_DEV_TIMEOUT);
                    }
                    break;
                }
                const uint32_t st = sbase + (uint32_t)s * STAGE_BYTES;
                const int nk = min(4, kmma_total - 4 * kt);
                // the scale factors first, on their own barrier, so the SF movers can
                // put them into tensor memory while the codes are still arriving;
                // boxes always deliver their full size (out-of-range parts are zero-filled)
                const uint32_t sfb_bytes = FMT ? 1024u : 4096u;
                const int sfb_row = (t.e * p.N + t.nt * 256) >> 7;
                if constexpr (CG == 2) {
                    // both CTAs' copies complete on the first CTA's barriers, which expect
                    // the bytes of both (a copy may land before the expectation: the phase
                    // cannot complete while the first CTA's arrival is pending).  The second
                    // CTA's rows are loaded even past the expert's segment (rows past the
                    // capacity read as zeros; rows of the next expert are never stored)
                    if (rank == 0) {
                        mbar_expect_tx_w(sf_full(s), 2u * (sfb_bytes + (FMT ? 512u : 2048u)));
                        mbar_expect_tx_w(full_bar(s), 2u * (16384u + 16384u));
                    }
                    if (swiglu)
                        tma_load_3d_w<2>(st + GM_SFB_OFF, &tmSFB, kt * 256, t.nt, 2 * t.e, lead(sf_full(s)));
                    else
                        tma_load_2d_w<2>(st + GM_SFB_OFF, &tmSFB, kt * (FMT ? 64 : 256), sfb_row, lead(sf_full(s)));
                    tma_load_2d_w<2>(st + GM_SFA_OFF, &tmSFA, kt * (FMT ? 64 : 256), my_m0 >> 7, lead(sf_full(s)));
                    tma_load_2d_w<2>(st + GM_A_OFF, &tmA, kt * 128, my_m0, lead(full_bar(s)));
                    // this CTA's half of B: the gate or the up row block (SwiGLU), else N rows 128r..
                    const int brow = swiglu ? t.e * p.N + (int)rank * (p.N >> 1) + t.nt * 128
                                            : t.e * p.N + t.nt * 256 + 128 * (int)rank;
                    tma_load_2d_w<2>(st + GM_B_OFF, &tmB, kt * 128, brow, lead(full_bar(s)));
                } else {
                    if constexpr (FMT == 1) {  // one chunk for A, one per B row tile
                        mbar_expect_tx_w(sf_full(s), sfb_bytes + 512u);
                        tma_load_2d_w(st + GM_SFB_OFF, &tmSFB, kt * 64, sfb_row, sf_full(s));
                        bulk_load_w(st + GM_SFA_OFF, sfa_src + (size_t)kt * 512, 512u, sf_full(s));
                    } else {
                        mbar_expect_tx_w(sf_full(s), sfb_bytes + (uint32_t)nk * 512u);
                        if (swiglu)
                            tma_load_3d_w(st + GM_SFB_OFF, &tmSFB, kt * 256, t.nt, 2 * t.e, sf_full(s));
                        else
                            tma_load_2d_w(st + GM_SFB_OFF, &tmSFB, kt * 256, sfb_row, sf_full(s));
                        bulk_load_w(st + GM_SFA_OFF, sfa_src + (size_t)kt * 2048, (uint32_t)nk * 512u, sf_full(s));
                    }
                    mbar_expect_tx_w(full_bar(s), 16384u + 32768u);
                    tma_load_2d_w(st + GM_A_OFF, &tmA, kt * 128, t.m0, full_bar(s));
                    if (swiglu)
                        tma_load_4d_w(st + GM_B_OFF, &tmB, kt * 128, t.nt * 128, 0, t.e, full_bar(s));
                    else
                        tma_load_2d_w(st + GM_B_OFF, &tmB, kt * 128, t.e * p.N + t.nt * 256, full_bar(s));
                }
            }
        }
        if (aborted_w(abort_flag)) {
            // let the copies already issued land before the CTA exits: they
            // complete within microseconds, so a bounded pause of ~1M cycles
            // covers them whichever CTA's barrier they signal
            const long long t0 = clock64();
            while (clock64() - t0 < (1ll << 20)) __nanosleep(1000);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer (first CTA, whole warp)
        if (rank == 0) {
            uint32_t it = 0, tc = 0;
            bool ready = false;  // stage `it` already seen complete (codes and scale factors)
            const uint64_t adesc0 = smem_desc(sbase + GM_A_OFF, 16, 1024, 2);
            const uint64_t bdesc0 = smem_desc(sbase + GM_B_OFF, 16, 1024, 2);
            for (int k = 0; !aborted_w(abort_flag); ++k, ++tc) {
                const int tile = tile_of(k);
                if (tile >= total_tiles) break;
                // only the tile's width matters here (no expert lookup: shared-memory
                // loads from this warp are slow while the copies stream in)
                const int nt = tile % p.n_tiles;
                const uint32_t n_w = (swiglu || CG == 2 || nt * 256 + 128 < p.N) ? 256u : 128u;
                const uint32_t idesc = FMT ? idesc_mxf8(n_w, 0u, 128u * CG) : idesc_nvf4(n_w, 128u * CG);
                // the epilogue (both CTAs') has taken the previous accumulator out of tensor memory
                if (!mbar_wait_w<CG == 2>(acc_empty, (tc & 1u) ^ 1u, abort_flag)) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        report(p.dev_status, BSQ_DEV_TIMEOUT);
                    }
                    break;
                }
                tc_fence_after();
                bool stop = false;
                for (int kt = 0; kt < kt_count; ++kt, ++it) {
                    const int s = (int)(it % STAGES);
                    const uint32_t ph = (it / STAGES) & 1u;
                    // codes landed (TMA, both CTAs) and scale factors staged in tensor
                    // memory; usually already seen by the previous stage's last MMA
                    if (!ready) {
                        bool ok = mbar_wait_w(full_bar(s), ph, abort_flag);
                        ok = ok && mbar_wait_w(sf_bar(s), ph, abort_flag);
                        if (!ok) {
                            if (lane == 0) {
                                *abort_flag = 1;
                                report(p.dev_status, BSQ_DEV_TIMEOUT);
                            }
                            stop = true;
                            break;
                        }
                    }
                    tc_fence_after();
                    const int nk = min(4, kmma_total - 4 * kt);
                    // descriptors advance 32 bytes (2 in the >>4 address field) per K step
                    const uint64_t ad = adesc0 + (uint64_t)s * (STAGE_BYTES >> 4);
                    const uint64_t bd = bdesc0 + (uint64_t)s * (STAGE_BYTES >> 4);
                    const uint32_t sf_col = tmem + GM_SF_RING + (uint32_t)s * GM_SF_STAGE_COLS;
                    // the next stage in ring order (the next tile's first after the last
                    // K stage), tested by the stage's last MMA
                    const uint32_t it1 = it + 1;
                    const int s1 = (int)(it1 % STAGES);
                    const uint32_t ph1 = (it1 / STAGES) & 1u;
                    uint32_t polled = 0;
                    // MXFP8: one scale column per operand half, byte j per MMA
                    auto id_of = [&](int j) { return FMT ? (idesc | ((uint32_t)j << 4) | ((uint32_t)j << 29)) : idesc; };
                    auto sfa_of = [&](int j) { return FMT ? sf_col : sf_col + 4u * (uint32_t)j; };
                    auto sfb_of = [&](int j) { return FMT ? sf_col + 16u : sf_col + 16u + 8u * (uint32_t)j; };
                    if (nk == 4) {
                        // a full stage, unrolled with compile-time K steps: a runtime step
                        // count around the MMAs measured ~45% slower issue
                        const uint32_t acc0 = kt > 0 ? 1u : 0u;
                        tc_mma_bs_w<FMT, CG>(tmem, ad, bd, id_of(0), sfa_of(0), sfb_of(0), acc0);
#pragma unroll
                        for (int j = 1; j < 3; ++j)
                            tc_mma_bs_w<FMT, CG>(tmem, ad + 2 * j, bd + 2 * j, id_of(j), sfa_of(j), sfb_of(j), 1u);
                        polled = tc_mma_bs_poll2_w<FMT, CG>(tmem, ad + 6, bd + 6, id_of(3), sfa_of(3), sfb_of(3), 1u,
                                                            full_bar(s1), ph1, sf_bar(s1), ph1);
                    } else {
                        // the K tail (K % 256 != 0): fewer MMAs, no poll
                        for (int j = 0; j < nk; ++j)
                            tc_mma_bs_w<FMT, CG>(tmem, ad + 2 * j, bd + 2 * j, id_of(j), sfa_of(j), sfb_of(j),
                                                 (kt > 0 || j > 0) ? 1u : 0u);
                    }
                    ready = __all_sync(0xFFFFFFFFu, polled == 3u);
                    tc_commit_w<CG>(empty_bar(s));  // with CG 2: both CTAs' producers
                }
                if (stop) break;
                tc_commit_w<CG>(acc_full);  // with CG 2: both CTAs' epilogues
            }
            // the drain: completes once every MMA issued here has completed
            tc_commit_all<CG>(drain_bar);
        }
        __syncwarp();
    } else if (warp < 2 + SF_WARPS) {
        // ------------------------------------------------------ scale factors -> tensor memory (first CTA)
        // A stage's scale factors go into the tensor-memory ring with
        // tcgen05.cp 32x128b.warpx4 (each 512-byte chunk lands in all four
        // lane quadrants, the layout the block-scaled MMA reads) in three
        // chunk runs: A's four chunks (columns 4j), B's first and second 128
        // rows (columns 16 + 8j and 20 + 8j).  The mover warps share a stage's
        // chunks evenly and each commits to the stage's SF barrier.  With CG 2
        // each copy moves both CTAs' chunks, each into its own tensor memory.
        const int w_sf = warp - 2;
        if (rank == 0) {
            uint32_t it = 0;
            for (int k = 0; !aborted_w(abort_flag); ++k) {
                if (tile_of(k) >= total_tiles) break;
                bool stop = false;
                for (int kt = 0; kt < kt_count; ++kt, ++it) {
                    const int s = (int)(it % STAGES);
                    const uint32_t ph = (it / STAGES) & 1u;
                    // implies the slot's previous scale factors were consumed: a producer
                    // refills a stage only after the MMAs that read it completed
                    if (!mbar_wait_w(sf_full(s), ph, abort_flag)) {
                        if (lane == 0) {
                            *abort_flag = 1;
                            report(p.dev_status, BSQ_DEV_TIMEOUT);
                        }
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    // the stage's chunks: run 0 = A's (columns 4j), runs 1 and 2 = B's first
                    // and second 128 rows (columns 16 + 8j and 20 + 8j); mover w copies
                    // chunks w, w + SF_WARPS, ...
                    constexpr int kChunks = FMT ? 3 : 12;
                    static_assert(kChunks % SF_WARPS == 0, "scale-factor chunks split evenly between movers");
#pragma unroll
                    for (int i = 0; i < kChunks / SF_WARPS; ++i) {  // a compile-time count keeps the issue fast
                        const int c = w_sf + SF_WARPS * i;
                        const int run = FMT ? c : c >> 2, j = FMT ? 0 : c & 3;
                        const uint32_t src = sbase + (uint32_t)s * STAGE_BYTES +
                                             (run == 0 ? GM_SFA_OFF : GM_SFB_OFF + (FMT ? 512 : 2048) * (run - 1)) +
                                             512u * (uint32_t)j;
                        const uint32_t dst = tmem + GM_SF_RING + (uint32_t)s * GM_SF_STAGE_COLS +
                                             (run == 0 ? 4u * (uint32_t)j : 16u + 4u * (uint32_t)(run - 1) + 8u * (uint32_t)j);
                        tc_cp_sf_w<CG>(dst, smem_desc(src, 16, 128, 0));
                    }
                    tc_commit_w<CG>(sf_bar(s), 1);  // the MMA issuer's barrier only
                }
                if (stop) break;
            }
            // every copy issued here lands before tensor memory is freed (both CTAs wait)
            tc_commit_all<CG>(sf_drain(w_sf));
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ epilogue (every CTA)
        const int q = warp & 3;                                  // tensor-memory lane quadrant
        const int part = (warp - 2 - SF_WARPS) >> 2;             // 0..3: which 64 columns (32 h for SwiGLU)
        const uint32_t tlane = tmem + ((uint32_t)(32 * q) << 16);
        uint8_t* stage_buf = smem + Cfg::EPI_OFF + (warp - 2 - SF_WARPS) * GM_EPI_WARP_BYTES;
        const uint32_t acc_empty_lead = lead(acc_empty);
        uint32_t tc = 0;
        bool broke = false;
        // fused quantization of h: the unit whose rows await quantization
        bool pend_valid = false;
        int pend_ub = 0, pend_row0 = 0;
        // a unit's h rows: this CTA's scratch (by unit parity) or, with keep_h, h itself
        auto unit_h = [&](int ub, int r0) {
            return p.keep_h ? static_cast<uint8_t*>(p.out) + (size_t)r0 * p.ldo * 2
                            : reinterpret_cast<uint8_t*>(p.h_scratch) + ((size_t)blockIdx.x * 2 + ub) * 128 * p.ldo * 2;
        };
        // The per-token NVFP4 quantization of a finished unit's 128 rows of h:
        // the 16 epilogue warps meet (every store of the unit's h is then
        // visible to all of them), then quantize (gm_quantize_h_rows)
        auto quantize_unit = [&](int ub, int r0) {
            __syncwarp();
            asm volatile("bar.sync 1, %0;" ::"n"(32 * GM_EPI_WARPS) : "memory");
            gm_quantize_h_rows<EPI == GM_EPI_SWIGLU_Q46>(s_hmax[ub], unit_h(ub, r0), p.ldo, p.N >> 5, r0, p.m_capacity,
                                                         p.q_codes, p.q_sf, p.q_scale,
                                                         2 * (warp - 2 - SF_WARPS) + (lane >> 4), lane & 15);
        };
        for (int k = 0;; ++k, ++tc) {
            const int tile = tile_of(k);
            if (tile >= total_tiles) {
                // after the last tile: the fused quantization's last unit
                if constexpr (fused) {
                    if (pend_valid) quantize_unit(pend_ub, pend_row0);
                }
                break;
            }
            const TileInfo t = tile_info(tile);
            const int row0 = t.m0 + 128 * (int)rank;  // this CTA's rows of the tile
            const int row = row0 + 32 * q + lane;
            const bool active = half_valid(t) && (swiglu || part < 2 * t.n_halves);
            // bf16 epilogue: the row's FP32 rescale t_tok * t_expert is loaded while
            // the tile's MMAs run, since the first half is rescaled before the
            // accumulator goes back (a load issued after the wait would hold up
            // the hand-off).  The other epilogues load it after the hand-off.
            const float s_early = (EPI == BSQ_EPI_BF16 && active && row < p.m_capacity)
                                      ? __fmul_rn(__ldg(p.a_scale + row), __ldg(p.b_scale + t.e))
                                      : 0.0f;
            const bool ok = mbar_wait(acc_full, tc & 1u, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, ok)) {
                if (lane == 0) {
                    *abort_flag = 1;
                    report(p.dev_status, BSQ_DEV_TIMEOUT);
                }
                broke = true;
                break;
            }
            tc_fence_after();
            auto hand_back = [&]() {  // accumulator handed back to the MMA warp
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (CG == 2)
                        mbar_arrive_cluster(acc_empty_lead);
                    else
                        mbar_arrive(acc_empty);
                }
            };
            if constexpr (EPI == BSQ_EPI_BF16) {
                // Both 32-column halves come out of tensor memory with one wait,
                // and the accumulator is handed back before anything else; the
                // packing, the staging and the stores (which may wait for the
                // previous store to drain) come after.
                const float s = s_early;
                uint32_t r[64];
                if (active) {
                    tc_ld32_issue(tlane + 64 * part, r);
                    tc_ld32_issue(tlane + 64 * part + 32, r + 32);
                    tc_ld_wait(r);
                }
                hand_back();
                if (!active) continue;
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    uint32_t pk[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        pk[j] = pack_bf16x2(__uint_as_float(r[32 * h2 + 2 * j]) * s,
                                            __uint_as_float(r[32 * h2 + 2 * j + 1]) * s);
                    stage_reuse(lane);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        stage_put(stage_buf, lane, c, pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                    stage_store(stage_buf, lane, &tmOut, t.nt * 256 + 64 * part + 32 * h2, row0 + 32 * q);
                }
                continue;
            }
            uint32_t r[64];
            if (active) {
                if (swiglu) {  // gate columns 32*part.., up columns 128 + 32*part..
                    tc_ld32_issue(tlane + 32 * part, r);
                    tc_ld32_issue(tlane + 128 + 32 * part, r + 32);
                } else {
                    tc_ld32_issue(tlane + 64 * part, r);
                    tc_ld32_issue(tlane + 64 * part + 32, r + 32);
                }
                tc_ld_wait(r);
            }
            hand_back();
            if (active) {
            const float s = (row < p.m_capacity) ? __fmul_rn(__ldg(p.a_scale + row), __ldg(p.b_scale + t.e)) : 0.0f;
            if constexpr (swiglu) {
                // 32 h values = 64 contiguous bytes of this thread's row, stored
                // from registers as two 32-byte sectors (or four 16-byte pieces
                // when the output is only 16-byte aligned)
                if constexpr (!fused) {
                    if (row < p.m_capacity) {
                        uint32_t w[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            w[j] = pack_bf16x2(swiglu1(__uint_as_float(r[2 * j]) * s, __uint_as_float(r[32 + 2 * j]) * s),
                                               swiglu1(__uint_as_float(r[2 * j + 1]) * s, __uint_as_float(r[33 + 2 * j]) * s));
                        uint8_t* d = static_cast<uint8_t*>(p.out) + ((size_t)row * p.ldo + t.nt * 128 + 32 * part) * 2;
                        st_row32(d, w, p.out_vec32);
                        st_row32(d + 32, w + 8, p.out_vec32);
                    }
                } else {
                    // h of this CTA's 128 rows goes to its scratch (double-buffered by
                    // unit; h kept whole in `out` for staged checks), and each row's
                    // running max |h|, over the bf16 values the quantizer will read,
                    // to shared memory
                    if (row < p.m_capacity) {
                        uint32_t w[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            w[j] = pack_bf16x2(swiglu1(__uint_as_float(r[2 * j]) * s, __uint_as_float(r[32 + 2 * j]) * s),
                                               swiglu1(__uint_as_float(r[2 * j + 1]) * s, __uint_as_float(r[33 + 2 * j]) * s));
                        uint32_t m = 0;
#pragma unroll
                        for (int j = 0; j < 16; ++j) m = absmax_bf16x2(m, w[j]);
                        atomicMax(&s_hmax[(k / p.n_tiles) & 1][32 * q + lane], fold_halves(m));
                        uint8_t* d = unit_h((k / p.n_tiles) & 1, row0) + ((size_t)(32 * q + lane) * p.ldo + t.nt * 128 + 32 * part) * 2;
                        st_row32(d, w, p.out_vec32);
                        st_row32(d + 32, w + 8, p.out_vec32);
                    }
                }
            } else if (row < p.m_capacity) {
                float4* d = reinterpret_cast<float4*>(static_cast<float*>(p.out) + (size_t)row * p.ldo + t.nt * 256 +
                                                      64 * part);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    d[i] = make_float4(__uint_as_float(r[4 * i]) * s, __uint_as_float(r[4 * i + 1]) * s,
                                       __uint_as_float(r[4 * i + 2]) * s, __uint_as_float(r[4 * i + 3]) * s);
            }
            }
            if constexpr (fused) {
                // A unit's rows are quantized during the next unit's first tile,
                // after its accumulator went back, so the MMAs keep running
                if (t.nt == 0 && pend_valid) quantize_unit(pend_ub, pend_row0);
                if (t.nt == 0) pend_valid = false;
                if (t.nt == p.n_tiles - 1) {
                    pend_valid = active;
                    pend_ub = (k / p.n_tiles) & 1;
                    pend_row0 = row0;
                }
            }
        }
        (void)broke;
        if constexpr (Cfg::STAGED) {
            if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
            __syncwarp();
        }
    }

    __syncwarp();  // every warp converged again (the cluster barrier below is .aligned)
    // Tensor memory is freed only after every MMA and scale-factor copy that
    // writes it has completed: the issuing threads committed their drains
    // (with CG 2 to both CTAs), waited for here with a bound.
    if (warp == 1) {
        if (lane == 0) {
            if (rank == 0 || CG == 2) {
                mbar_drain(drain_bar, 0u);
                for (int w = 0; w < SF_WARPS; ++w) mbar_drain(sf_drain(w), 0u);
            }
        }
        __syncwarp();
    }
    tc_fence_before();
    if constexpr (CG == 2)
        cluster_sync();
    else
        __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem, GM_TMEM_COLS);
    }
    if constexpr (CG == 2) cluster_sync();  // neither CTA leaves while the pair still shares memory
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

// Tensor map of `rank` dims (dims/box innermost first, strides in bytes for
// dims 1..rank-1).
static bool make_tmap(CUtensorMap* tm, const void* base, CUtensorMapDataType dt, int rank, const cuuint64_t* dims,
                      const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
    return fn(tm, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EPI, int FMT, int CG>
static cudaError_t set_smem_attr()
{
    return cudaFuncSetAttribute(k_gemm_fp4<EPI, FMT, CG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)GmCfg<EPI, CG>::SMEM_BYTES);
}

template <int EPI, int FMT, int CG>
static cudaError_t launch_kernel(int64_t grid, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmSFA,
                                 const CUtensorMap& tmSFB, const CUtensorMap& tmOut, const GemmParams& p,
                                 cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(GmCfg<EPI, CG>::THREADS);
    cfg.dynamicSmemBytes = GmCfg<EPI, CG>::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_gemm_fp4<EPI, FMT, CG>, tmA, tmB, tmSFA, tmSFB, tmOut, p);
}

template <int CG>
static cudaError_t launch_form(const GemmArgs& a, int64_t grid, const CUtensorMap& tmA, const CUtensorMap& tmB,
                               const CUtensorMap& tmSFA, const CUtensorMap& tmSFB, const CUtensorMap& tmOut,
                               const GemmParams& p, cudaStream_t st)
{
    if (a.fmt == 1)
        return a.epilogue == BSQ_EPI_BF16
                   ? launch_kernel<BSQ_EPI_BF16, 1, CG>(grid, tmA, tmB, tmSFA, tmSFB, tmOut, p, st)
                   : launch_kernel<BSQ_EPI_F32, 1, CG>(grid, tmA, tmB, tmSFA, tmSFB, tmOut, p, st);
    if (a.epilogue == BSQ_EPI_SWIGLU_BF16)
        return launch_kernel<BSQ_EPI_SWIGLU_BF16, 0, CG>(grid, tmA, tmB, tmSFA, tmSFB, tmOut, p, st);
    if (a.epilogue == GM_EPI_SWIGLU_Q) return launch_kernel<GM_EPI_SWIGLU_Q, 0, CG>(grid, tmA, tmB, tmSFA, tmSFB, tmOut, p, st);
    if (a.epilogue == GM_EPI_SWIGLU_Q46)
        return launch_kernel<GM_EPI_SWIGLU_Q46, 0, CG>(grid, tmA, tmB, tmSFA, tmSFB, tmOut, p, st);
    if (a.epilogue == BSQ_EPI_BF16) return launch_kernel<BSQ_EPI_BF16, 0, CG>(grid, tmA, tmB, tmSFA, tmSFB, tmOut, p, st);
    return launch_kernel<BSQ_EPI_F32, 0, CG>(grid, tmA, tmB, tmSFA, tmSFB, tmOut, p, st);
}

template <int CG>
static cudaError_t set_form_attrs()
{
    cudaError_t err = set_smem_attr<BSQ_EPI_F32, 0, CG>();
    if (err == cudaSuccess) err = set_smem_attr<BSQ_EPI_BF16, 0, CG>();
    if (err == cudaSuccess) err = set_smem_attr<BSQ_EPI_SWIGLU_BF16, 0, CG>();
    if (err == cudaSuccess) err = set_smem_attr<GM_EPI_SWIGLU_Q, 0, CG>();
    if (err == cudaSuccess) err = set_smem_attr<GM_EPI_SWIGLU_Q46, 0, CG>();
    if (err == cudaSuccess) err = set_smem_attr<BSQ_EPI_F32, 1, CG>();
    if (err == cudaSuccess) err = set_smem_attr<BSQ_EPI_BF16, 1, CG>();
    return err;
}

// The form and the CTAs a launch uses (the pair form keeps every expert's
// first pair tile in shared memory).
static int gemm_form(int64_t experts, int sms) { return experts <= GM_MAX_SMEM_EXPERTS && sms >= 2 ? 2 : 1; }
int64_t gemm_fp4_ctas(int64_t experts, int64_t m_capacity, int64_t n_tiles, int sms)
{
    const int64_t max_units = ((m_capacity + 127) / 128) * n_tiles;
    if (gemm_form(experts, sms) == 2) return 2 * std::min<int64_t>(max_units, sms / 2);
    return std::min<int64_t>(max_units, sms);
}

cudaError_t launch_gemm_fp4(const GemmArgs& a, cudaStream_t st)
{
    static std::atomic<uint64_t> attr_done{0};
    cudaError_t aerr = once_per_device(attr_done, [] {
        cudaError_t err = set_form_attrs<1>();
        return err == cudaSuccess ? set_form_attrs<2>() : err;
    });
    if (aerr != cudaSuccess) return aerr;
    const bool fused = a.epilogue == GM_EPI_SWIGLU_Q || a.epilogue == GM_EPI_SWIGLU_Q46;
    const bool swiglu = a.epilogue == BSQ_EPI_SWIGLU_BF16 || fused;
    const bool mx8 = a.fmt == 1;                 // MXFP8 operands (no SwiGLU epilogue)
    if (fused && (!a.q_codes || !a.q_sf || !a.q_scale || (!a.keep_h && !a.h_scratch))) return cudaErrorInvalidValue;
    if (mx8 && swiglu) return cudaErrorInvalidValue;
    const int cg = gemm_form(a.experts, a.sms);
    const int64_t kb = mx8 ? a.K : a.K / 2;      // bytes per row of codes
    const int64_t k64 = mx8 ? a.K / 128 : a.K / 64;  // 512-byte SF chunks per row tile
    const int64_t m_tiles = (a.m_capacity + 127) / 128;
    CUtensorMap tmA, tmB, tmSFA, tmSFB;
    memset(&tmSFA, 0, sizeof(tmSFA));
    {   // A: [m_capacity][K/2] bytes, box 128 x 128
        const cuuint64_t d[2] = {(cuuint64_t)kb, (cuuint64_t)a.m_capacity};
        const cuuint64_t s[1] = {(cuuint64_t)kb};
        const cuuint32_t b[2] = {128u, 128u};
        if (!make_tmap(&tmA, a.a_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    if (cg == 2) {
        // B: [E*N rows][K/2] bytes, box 128 x 128: each CTA of a pair loads one 128-row half
        const cuuint64_t d[2] = {(cuuint64_t)kb, (cuuint64_t)(a.experts * a.N)};
        const cuuint64_t s[1] = {(cuuint64_t)kb};
        const cuuint32_t b[2] = {128u, 128u};
        if (!make_tmap(&tmB, a.b_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        // A's SF as u64 [row tiles][k64 * 64]: one box = a row tile's stage run (2 KB NVFP4, 512 B MXFP8)
        const cuuint64_t sd[2] = {(cuuint64_t)(k64 * 64), (cuuint64_t)m_tiles};
        const cuuint64_t ss[1] = {(cuuint64_t)(k64 * 512)};
        const cuuint32_t sb[2] = {mx8 ? 64u : 256u, 1u};
        if (!make_tmap(&tmSFA, a.a_sf, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, sd, ss, sb, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else if (swiglu) {
        // B viewed as [E][2 (gate, up)][I rows][K/2 bytes]: one box = 128 gate + 128 up rows
        const int64_t I = a.N / 2;
        const cuuint64_t d[4] = {(cuuint64_t)kb, (cuuint64_t)I, 2u, (cuuint64_t)a.experts};
        const cuuint64_t s[3] = {(cuuint64_t)kb, (cuuint64_t)(I * kb), (cuuint64_t)(2 * I * kb)};
        const cuuint32_t b[4] = {128u, 128u, 2u, 1u};
        if (!make_tmap(&tmB, a.b_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    } else {
        const cuuint64_t d[2] = {(cuuint64_t)kb, (cuuint64_t)(a.experts * a.N)};
        const cuuint64_t s[1] = {(cuuint64_t)kb};
        const cuuint32_t b[2] = {128u, 256u};
        if (!make_tmap(&tmB, a.b_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    if (swiglu) {
        // B's SF as u64 [E * 2 (gate, up)][I/128 row tiles][k64 * 64]: one box = the
        // 2 KB stage run of the gate row tile and of the up row tile
        const int64_t I = a.N / 2;
        const cuuint64_t sd[3] = {(cuuint64_t)(k64 * 64), (cuuint64_t)(I / 128), (cuuint64_t)(2 * a.experts)};
        const cuuint64_t ss[2] = {(cuuint64_t)(k64 * 512), (cuuint64_t)((I / 128) * k64 * 512)};
        const cuuint32_t sb[3] = {256u, 1u, 2u};
        if (!make_tmap(&tmSFB, a.b_sf, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, sd, ss, sb, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else {
        // B's SF as u64 [E*N/128 row tiles][k64 * 64]: one box = the stage runs of two row tiles
        // (2 KB each for NVFP4, 512 bytes for MXFP8)
        const cuuint64_t sd[2] = {(cuuint64_t)(k64 * 64), (cuuint64_t)(a.experts * a.N / 128)};
        const cuuint64_t ss[1] = {(cuuint64_t)(k64 * 512)};
        const cuuint32_t sb[2] = {mx8 ? 64u : 256u, 2u};
        if (!make_tmap(&tmSFB, a.b_sf, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, sd, ss, sb, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    CUtensorMap tmOut;
    if (a.epilogue != BSQ_EPI_BF16) {
        memset(&tmOut, 0, sizeof(tmOut));  // f32 and SwiGLU outputs are stored from registers
    } else {
        // bf16 output [m_capacity][N] with row pitch ldo: 32 x 32 boxes, 64-byte swizzle
        const int64_t ncols = a.N;
        const cuuint64_t d[2] = {(cuuint64_t)ncols, (cuuint64_t)a.m_capacity};
        const cuuint64_t s[1] = {(cuuint64_t)(a.ldo * 2)};
        const cuuint32_t b[2] = {32u, 32u};
        if (!make_tmap(&tmOut, a.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, s, b, CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    }
    GemmParams p;
    p.a_sf = a.a_sf;
    p.b_sf = a.b_sf;
    p.a_scale = a.a_scale;
    p.offsets = a.offsets;
    p.b_scale = a.b_scale;
    p.out = a.out;
    p.dev_status = a.dev_status;
    p.ldo = a.ldo;
    p.experts = (int32_t)a.experts;
    p.m_capacity = (int32_t)a.m_capacity;
    p.K = (int32_t)a.K;
    p.N = (int32_t)a.N;
    p.epilogue = a.epilogue;
    p.out_vec32 = (reinterpret_cast<uintptr_t>(fused && !a.keep_h ? (const void*)a.h_scratch : a.out) % 32 == 0) &&
                  ((a.ldo * 2) % 32 == 0);
    p.q_codes = a.q_codes;
    p.q_sf = a.q_sf;
    p.q_scale = a.q_scale;
    p.h_scratch = a.h_scratch;
    p.keep_h = a.keep_h;
    p.n_tiles = swiglu ? (int32_t)(a.N / 256) : (int32_t)((a.N + 255) / 256);
    // persistent: at most one CTA per SM, never more CTAs (or pairs) than the largest
    // possible tile count (a pair tile covers at least one 128-row tile)
    const int64_t max_units = m_tiles * p.n_tiles;
    if (cg == 2) {
        const int64_t pairs = std::min<int64_t>(max_units, a.sms / 2);
        if (pairs <= 0) return cudaSuccess;
        cudaError_t err = launch_form<2>(a, 2 * pairs, tmA, tmB, tmSFA, tmSFB, tmOut, p, st);
        return err != cudaSuccess ? err : cudaGetLastError();
    }
    const int64_t grid = std::min<int64_t>(max_units, a.sms);
    if (grid <= 0) return cudaSuccess;
    cudaError_t err = launch_form<1>(a, grid, tmA, tmB, tmSFA, tmSFB, tmOut, p, st);
    return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace bsq
