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
// meccanismo"); on GB300 the FP4 tensor cores are fast enough that feeding
// them is the hard part ("End-to-End 4-Bit Training", section "工程细节").
//
// Persistent kernel, one CTA per SM.  The grouped problem is flattened into
// 128-row x 256-column output tiles (128-row tiles of the expert-sorted A,
// each inside one expert's segment, times the N tiles), walked round-robin.
// One 128 x 256 x 64 FP4 MMA occupies the tensor core for 128 cycles, so a
// 256-wide K stage (4 MMAs, 54 KB of operands and scale factors) must arrive
// every ~512 cycles: the kernel is fed by the TMA engine at close to its
// per-SM rate, and everything else is arranged to stay off that path.
//   warp 0      TMA producer.  Per stage it first copies the scale factors
//               (A's: one 2 KB bulk copy; B's: two 512-byte-chunk runs in one
//               2-D/3-D box of u64 elements) on their own barrier, then the
//               codes: A (128 x 128 B) and B (256 rows: one 2-D box, or the
//               gate + up blocks in one 4-D box for SwiGLU)
//   warp 1      allocates tensor memory; one lane issues one 128 x 256 x 64
//               MMA per K step and the commits.  It touches shared memory only
//               for its barrier waits (a tile's width is all it needs to know)
//   warps 2..   one or three scale-factor movers: as soon as a stage's scale
//               factors land, they are copied into tensor memory with
//               tcgen05.cp 32x128b.warpx4 while the codes are still in flight
//               (each 512-byte chunk lands replicated in all four lane
//               quadrants)
//   the last 16 warps  epilogue, four per lane quadrant, 64 columns each: load
//               the accumulator, hand it back to the MMA warp, then rescale /
//               SwiGLU / store while the next tile's MMAs run
// Shared memory: a ring of stages of [SFA 2 KB][SFB 4 KB][A 16 KB][B 32 KB]
// (A and B 128-byte swizzled, 1024-byte aligned) and the expert offsets.  The
// ring's depth is what hides the round trip of a stage (MMAs complete ->
// stage released -> copies issued -> copies landed: ~2700 cycles against 512
// cycles of MMAs per stage), so every epilogue that can store straight from
// registers gets four stages.  Only the plain bf16 epilogue, whose 128 x 256
// output tile is the largest, keeps three stages plus a 2 KB staging buffer
// per epilogue warp: a warp writes each 32 x 32 block of its 32 rows there
// and one lane stores it with a TMA tensor store.
// Tensor memory: 512 columns = accumulator (256) + an SF ring (48 per stage:
// SFA k-step j at 4j, SFB k-step j at 16 + 8j, both N halves side by side).
// Every mbarrier wait is bounded; on expiry the CTA records BSQ_DEV_TIMEOUT,
// drains its outstanding copies and MMAs (bounded), frees tensor memory and
// returns.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace bsq {

constexpr int GM_MAX_SF_WARPS = 3;
constexpr int GM_EPI_WARPS = 16;
constexpr int GM_MAX_STAGES = 4;
constexpr int GM_SFA_OFF = 0;
constexpr int GM_SFB_OFF = 2048;
constexpr int GM_A_OFF = 6144;
constexpr int GM_B_OFF = 6144 + 16384;
constexpr int GM_STAGE_BYTES = 6144 + 16384 + 32768;  // 55296 = 54 KB
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
constexpr int GM_EPI_WARP_BYTES = 32 * 64;                     // 32 rows x 64 bytes, 64-byte swizzled

// Per epilogue kind: the stage count, whether the epilogue stages its stores
// through shared memory (after the ring), the dynamic shared memory, and the
// number of scale-factor mover warps.  Three movers (one chunk run each) get
// each stage's scale factors into tensor memory soonest, which the four-stage
// SwiGLU GEMM, bound by the stage round trip, needs; one mover keeps the CTA
// at 19 warps, at most five per SM sub-partition and 96 registers a thread,
// which lets the epilogue warps that share a sub-partition with the producer
// hand the accumulator back in time on the short-K bf16 GEMM.
template <int EPI>
struct GmCfg {
    static constexpr int SF_WARPS = EPI == BSQ_EPI_SWIGLU_BF16 ? 3 : 1;
    static constexpr int THREADS = 32 * (2 + SF_WARPS + GM_EPI_WARPS);
    static constexpr bool STAGED = EPI == BSQ_EPI_BF16;
    static constexpr int STAGES = STAGED ? 3 : 4;
    static constexpr int EPI_OFF = STAGES * GM_STAGE_BYTES;
    static constexpr size_t SMEM_BYTES =
        (size_t)EPI_OFF + (STAGED ? (size_t)GM_EPI_WARPS * GM_EPI_WARP_BYTES : 0) + 1024;
};
static_assert(GM_SF_RING + GM_MAX_STAGES * GM_SF_STAGE_COLS <= GM_TMEM_COLS, "SF ring exceeds tensor memory");
static_assert(GmCfg<BSQ_EPI_SWIGLU_BF16>::SMEM_BYTES + 2048 <= 232448, "stage ring exceeds shared memory");

// Bounded wait; gives up when the abort flag is raised or the spin limit hit.
BSQ_DEVICE bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag)
{
    for (uint32_t i = 0; i < GM_SPIN_LIMIT; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && *abort_flag) return false;
    }
    return false;
}

BSQ_DEVICE uint32_t pack_bf16x2(float lo, float hi)
{
    const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return l | (h << 16);
}


// h = silu(g) * u with silu(g) = g / (1 + e^-g); approximate exponential and
// division (relative error ~1e-6, far below the bf16 output rounding); the
// e^-g -> inf limit gives h -> 0.
BSQ_DEVICE float swiglu1(float g, float u) { return __fdividef(g * u, 1.0f + __expf(-g)); }

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
};

struct TileInfo {
    int m0, nt, e, n_halves;
};

// EPI is the epilogue (BSQ_EPI_*): one instantiation per epilogue keeps each
// one's register allocation to its own path.  FMT is the operand format:
// 0 NVFP4 (E2M1 codes, E4M3 scale per 16, kind::mxf4nvf4, K = 64 per MMA,
// four 512-byte scale chunks per 128 rows and stage), 1 MXFP8 (E4M3 codes,
// E8M0 scale per 32, kind::mxf8f6f4, K = 32 per MMA, one chunk per 128 rows
// and stage).  A stage is 128 bytes of every row in both.
template <int EPI, int FMT = 0>
__global__ void __launch_bounds__(GmCfg<EPI>::THREADS, 1)
    k_gemm_fp4(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmSFB, const __grid_constant__ CUtensorMap tmOut,
               const GemmParams p)
{
    constexpr int GM_STAGES = GmCfg<EPI>::STAGES;
    constexpr int GM_SF_WARPS = GmCfg<EPI>::SF_WARPS;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[4 * GM_MAX_STAGES + 3 + GM_MAX_SF_WARPS];
    __shared__ int32_t s_off[GM_MAX_SMEM_EXPERTS + 1];
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort, s_bad;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.experts;
    const bool off_in_smem = E <= GM_MAX_SMEM_EXPERTS;
    for (int i = threadIdx.x; i <= E && off_in_smem; i += blockDim.x) s_off[i] = __ldg(p.offsets + i);

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(GM_STAGES + s); };
    auto sf_bar = [&](int s) { return bar0 + 8u * (uint32_t)(2 * GM_STAGES + s); };
    auto sf_full = [&](int s) { return bar0 + 8u * (uint32_t)(3 * GM_STAGES + s); };
    const uint32_t acc_full = bar0 + 8u * (4 * GM_STAGES);
    const uint32_t acc_empty = bar0 + 8u * (4 * GM_STAGES + 1);
    const uint32_t drain_bar = bar0 + 8u * (4 * GM_STAGES + 2);
    auto sf_drain = [&](int w) { return bar0 + 8u * (uint32_t)(4 * GM_STAGES + 3 + w); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < GM_STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
            mbar_init(sf_bar(s), GM_SF_WARPS);
            mbar_init(sf_full(s), 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, GM_EPI_WARPS);
        mbar_init(drain_bar, 1);
        for (int w = 0; w < GM_SF_WARPS; ++w) mbar_init(sf_drain(w), 1);
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
        if (bad) report(p.dev_status, BSQ_DEV_BAD_OFFSETS);
    }
    __syncthreads();

    constexpr bool swiglu = EPI == BSQ_EPI_SWIGLU_BF16;
    const int kmma_total = FMT ? (p.K >> 5) : (p.K >> 6);  // MMAs along K (64 or 32 elements each)
    const int kt_count = (kmma_total + 3) >> 2;
    const int sf_chunks = FMT ? (p.K >> 7) : (p.K >> 6);  // 512-byte scale chunks per 128-row tile
    const int m_tiles = s_bad ? 0 : (off(E) + 127) >> 7;
    const int total_tiles = m_tiles * p.n_tiles;

    auto tile_info = [&](int tile) {
        TileInfo t;
        t.nt = tile % p.n_tiles;
        t.m0 = (tile / p.n_tiles) * 128;
        int lo = 0, hi = E - 1;  // largest e with offsets[e] <= m0
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (off(mid) <= t.m0) lo = mid; else hi = mid - 1;
        }
        t.e = lo;
        t.n_halves = swiglu ? 2 : ((t.nt * 256 + 128 < p.N) ? 2 : 1);
        return t;
    };

    if (warp == 0) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmSFB)) : "memory");
            uint32_t it = 0;
            for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag && !GM_STALL; tile += gridDim.x) {
                const TileInfo t = tile_info(tile);
                const uint8_t* sfa_src = p.a_sf + ((size_t)(t.m0 >> 7) * sf_chunks) * 512;
                for (int kt = 0; kt < kt_count; ++kt, ++it) {
                    const int s = (int)(it % GM_STAGES);
                    const uint32_t ph = (it / GM_STAGES) & 1u;
                    if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag)) {
                        *abort_flag = 1;
                        report(p.dev_status, BSQ_DEV_TIMEOUT);
                        break;
                    }
                    const uint32_t st = sbase + (uint32_t)s * GM_STAGE_BYTES;
                    const int nk = min(4, kmma_total - 4 * kt);
                    // the scale factors first, on their own barrier, so the SF warps can
                    // move them into tensor memory while the codes are still arriving;
                    // boxes always deliver their full size (out-of-range parts are zero-filled)
                    if constexpr (FMT == 1) {  // one chunk for A, one per B row tile
                        mbar_expect_tx(sf_full(s), 1024u + 512u);
                        tma_load_2d(st + GM_SFB_OFF, &tmSFB, kt * 64, (t.e * p.N + t.nt * 256) >> 7, sf_full(s));
                        bulk_load(st + GM_SFA_OFF, sfa_src + (size_t)kt * 512, 512u, sf_full(s));
                    } else {
                        mbar_expect_tx(sf_full(s), 4096u + (uint32_t)nk * 512u);
                        if (swiglu)
                            tma_load_3d(st + GM_SFB_OFF, &tmSFB, kt * 256, t.nt, 2 * t.e, sf_full(s));
                        else
                            tma_load_2d(st + GM_SFB_OFF, &tmSFB, kt * 256, (t.e * p.N + t.nt * 256) >> 7, sf_full(s));
                        bulk_load(st + GM_SFA_OFF, sfa_src + (size_t)kt * 2048, (uint32_t)nk * 512u, sf_full(s));
                    }
                    mbar_expect_tx(full_bar(s), 16384u + 32768u);
                    tma_load_2d(st + GM_A_OFF, &tmA, kt * 128, t.m0, full_bar(s));
                    if (swiglu)
                        tma_load_4d(st + GM_B_OFF, &tmB, kt * 128, t.nt * 128, 0, t.e, full_bar(s));
                    else
                        tma_load_2d(st + GM_B_OFF, &tmB, kt * 128, t.e * p.N + t.nt * 256, full_bar(s));
                }
            }
            if (*abort_flag) {
                // let the copies already issued land before the CTA exits
                for (uint32_t j = (it > GM_STAGES ? it - GM_STAGES : 0u); j < it; ++j) {
                    for (uint32_t i = 0; i < GM_SPIN_LIMIT; ++i)
                        if (mbar_try_wait(full_bar((int)(j % GM_STAGES)), (j / GM_STAGES) & 1u)) break;
                    for (uint32_t i = 0; i < GM_SPIN_LIMIT; ++i)
                        if (mbar_try_wait(sf_full((int)(j % GM_STAGES)), (j / GM_STAGES) & 1u)) break;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, tc = 0;
            bool issued_any = false;
            const uint64_t adesc0 = smem_desc(sbase + GM_A_OFF, 16, 1024, 2);
            const uint64_t bdesc0 = smem_desc(sbase + GM_B_OFF, 16, 1024, 2);
            for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x, ++tc) {
                // only the tile's width matters here (no expert lookup: shared-memory
                // loads from this thread are slow while the copies stream in)
                const int nt = tile % p.n_tiles;
                const uint32_t n_w = (swiglu || nt * 256 + 128 < p.N) ? 256u : 128u;
                const uint32_t idesc = FMT ? idesc_mxf8(n_w, 0u) : idesc_nvf4(n_w);
                // the epilogue has taken the previous accumulator out of tensor memory
                if (!mbar_wait(acc_empty, (tc & 1u) ^ 1u, abort_flag)) {
                    *abort_flag = 1;
                    report(p.dev_status, BSQ_DEV_TIMEOUT);
                    break;
                }
                tc_fence_after();
                for (int kt = 0; kt < kt_count; ++kt, ++it) {
                    const int s = (int)(it % GM_STAGES);
                    const uint32_t ph = (it / GM_STAGES) & 1u;
                    // codes landed (TMA) and scale factors staged in tensor memory (SF warps)
                    bool ok = mbar_wait(full_bar(s), ph, abort_flag);
                    ok = ok && mbar_wait(sf_bar(s), ph, abort_flag);
                    if (!ok) {
                        *abort_flag = 1;
                        report(p.dev_status, BSQ_DEV_TIMEOUT);
                        break;
                    }
                    tc_fence_after();
                    const int nk = min(4, kmma_total - 4 * kt);
                    // descriptors advance 32 bytes (2 in the >>4 address field) per K step
                    const uint64_t ad = adesc0 + (uint64_t)s * (GM_STAGE_BYTES >> 4);
                    const uint64_t bd = bdesc0 + (uint64_t)s * (GM_STAGE_BYTES >> 4);
                    const uint32_t sf_col = tmem + GM_SF_RING + (uint32_t)s * GM_SF_STAGE_COLS;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (j < nk) {
                            if constexpr (FMT == 1)  // one scale column per operand half; byte j per MMA
                                tc_mma_bs<1>(tmem, ad + 2 * j, bd + 2 * j, idesc | ((uint32_t)j << 4) | ((uint32_t)j << 29),
                                           sf_col, sf_col + 16, (kt > 0 || j > 0) ? 1u : 0u);
                            else
                                tc_mma_bs<0>(tmem, ad + 2 * j, bd + 2 * j, idesc, sf_col + 4 * j, sf_col + 16 + 8 * j,
                                       (kt > 0 || j > 0) ? 1u : 0u);
                        }
                    tc_commit(empty_bar(s));
                    issued_any = true;
                }
                if (*abort_flag) break;
                tc_commit(acc_full);
            }
            // tensor memory is freed only after every MMA issued here has completed
            if (issued_any) {
                tc_commit(drain_bar);
                for (uint32_t i = 0; i < GM_SPIN_LIMIT; ++i)
                    if (mbar_try_wait(drain_bar, 0u)) break;
            }
        }
        __syncwarp();
    } else if (warp < 2 + GM_SF_WARPS) {
        // ------------------------------------------------------ scale factors -> tensor memory
        // A stage's scale factors go into the tensor-memory ring with
        // tcgen05.cp 32x128b.warpx4 (each 512-byte chunk lands in all four
        // lane quadrants, the layout the block-scaled MMA reads) in three
        // chunk runs: A's four chunks (columns 4j), B's first and second 128
        // rows (columns 16 + 8j and 20 + 8j).  With three mover warps, lane 0
        // of warp 2 + r moves run r; with one, lane 0 of warp 2 moves all
        // three.  Each then commits to the stage's SF barrier.  The copies
        // start as soon as the SF land, while the codes are still in flight,
        // and they neither pass through registers nor cost shared-memory
        // reads beyond the 6 KB themselves.
        const int w_sf = warp - 2;
        const int run0 = GM_SF_WARPS == 1 ? 0 : w_sf, run1 = GM_SF_WARPS == 1 ? 3 : w_sf + 1;
        if (lane == 0) {
            uint32_t it = 0;
            for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
                for (int kt = 0; kt < kt_count; ++kt, ++it) {
                    const int s = (int)(it % GM_STAGES);
                    const uint32_t ph = (it / GM_STAGES) & 1u;
                    // implies the slot's previous scale factors were consumed: the producer
                    // refills a stage only after the MMAs that read it completed
                    if (!mbar_wait(sf_full(s), ph, abort_flag)) {
                        *abort_flag = 1;
                        report(p.dev_status, BSQ_DEV_TIMEOUT);
                        break;
                    }
                    tc_fence_after();
                    for (int run = run0; run < run1; ++run) {
                        const uint32_t src = sbase + (uint32_t)s * GM_STAGE_BYTES +
                                             (run == 0 ? GM_SFA_OFF : GM_SFB_OFF + (FMT ? 512 : 2048) * (run - 1));
                        const uint32_t dst = tmem + GM_SF_RING + (uint32_t)s * GM_SF_STAGE_COLS +
                                             (run == 0 ? 0u : 16u + 4u * (uint32_t)(run - 1));
                        const uint32_t step = run == 0 ? 4u : 8u;
#pragma unroll
                        for (int j = 0; j < (FMT ? 1 : 4); ++j)
                            tc_cp_sf(dst + step * j, smem_desc(src + 512 * j, 16, 128, 0));
                    }
                    tc_commit(sf_bar(s));
                }
            }
            // every copy issued here lands before tensor memory is freed
            tc_commit(sf_drain(w_sf));
            for (uint32_t i = 0; i < GM_SPIN_LIMIT; ++i)
                if (mbar_try_wait(sf_drain(w_sf), 0u)) break;
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;                                  // tensor-memory lane quadrant
        const int part = (warp - 2 - GM_SF_WARPS) >> 2;          // 0..3: which 64 columns (32 h for SwiGLU)
        const uint32_t tlane = tmem + ((uint32_t)(32 * q) << 16);
        uint8_t* stage_buf = smem + GmCfg<EPI>::EPI_OFF + (warp - 2 - GM_SF_WARPS) * GM_EPI_WARP_BYTES;
        uint32_t tc = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++tc) {
            const TileInfo t = tile_info(tile);
            const int row = t.m0 + 32 * q + lane;
            const bool active = swiglu || part < 2 * t.n_halves;
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
                break;
            }
            tc_fence_after();
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
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
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
                    stage_store(stage_buf, lane, &tmOut, t.nt * 256 + 64 * part + 32 * h2, t.m0 + 32 * q);
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
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);  // accumulator handed back to the MMA warp
            if (!active) continue;
            const float s = (row < p.m_capacity) ? __fmul_rn(__ldg(p.a_scale + row), __ldg(p.b_scale + t.e)) : 0.0f;
            if constexpr (swiglu) {
                // 32 h values = 64 contiguous bytes of this thread's row, stored
                // from registers as two 32-byte sectors (or four 16-byte pieces
                // when the output is only 16-byte aligned)
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
            } else if (row < p.m_capacity) {
                float4* d = reinterpret_cast<float4*>(static_cast<float*>(p.out) + (size_t)row * p.ldo + t.nt * 256 +
                                                      64 * part);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    d[i] = make_float4(__uint_as_float(r[4 * i]) * s, __uint_as_float(r[4 * i + 1]) * s,
                                       __uint_as_float(r[4 * i + 2]) * s, __uint_as_float(r[4 * i + 3]) * s);
            }
        }
        if constexpr (GmCfg<EPI>::STAGED) {
            if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
            __syncwarp();
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

cudaError_t launch_gemm_fp4(const GemmArgs& a, cudaStream_t st)
{
    static std::atomic<uint64_t> attr_done{0};
    cudaError_t aerr = once_per_device(attr_done, [] {
        cudaError_t err = cudaFuncSetAttribute(k_gemm_fp4<BSQ_EPI_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)GmCfg<BSQ_EPI_F32>::SMEM_BYTES);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(k_gemm_fp4<BSQ_EPI_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)GmCfg<BSQ_EPI_BF16>::SMEM_BYTES);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(k_gemm_fp4<BSQ_EPI_SWIGLU_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)GmCfg<BSQ_EPI_SWIGLU_BF16>::SMEM_BYTES);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(k_gemm_fp4<BSQ_EPI_F32, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)GmCfg<BSQ_EPI_F32>::SMEM_BYTES);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(k_gemm_fp4<BSQ_EPI_BF16, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)GmCfg<BSQ_EPI_BF16>::SMEM_BYTES);
        return err;
    });
    if (aerr != cudaSuccess) return aerr;
    const bool swiglu = a.epilogue == BSQ_EPI_SWIGLU_BF16;
    const bool mx8 = a.fmt == 1;                 // MXFP8 operands (no SwiGLU epilogue)
    if (mx8 && swiglu) return cudaErrorInvalidValue;
    const int64_t kb = mx8 ? a.K : a.K / 2;      // bytes per row of codes
    const int64_t k64 = mx8 ? a.K / 128 : a.K / 64;  // 512-byte SF chunks per row tile
    CUtensorMap tmA, tmB, tmSFB;
    {   // A: [m_capacity][K/2] bytes, box 128 x 128
        const cuuint64_t d[2] = {(cuuint64_t)kb, (cuuint64_t)a.m_capacity};
        const cuuint64_t s[1] = {(cuuint64_t)kb};
        const cuuint32_t b[2] = {128u, 128u};
        if (!make_tmap(&tmA, a.a_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    if (swiglu) {
        // B viewed as [E][2 (gate, up)][I rows][K/2 bytes]: one box = 128 gate + 128 up rows
        const int64_t I = a.N / 2;
        const cuuint64_t d[4] = {(cuuint64_t)kb, (cuuint64_t)I, 2u, (cuuint64_t)a.experts};
        const cuuint64_t s[3] = {(cuuint64_t)kb, (cuuint64_t)(I * kb), (cuuint64_t)(2 * I * kb)};
        const cuuint32_t b[4] = {128u, 128u, 2u, 1u};
        if (!make_tmap(&tmB, a.b_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        // B's SF as u64 [E * 2 (gate, up)][I/128 row tiles][k64 * 64]: one box = the
        // 2 KB stage run of the gate row tile and of the up row tile
        const cuuint64_t sd[3] = {(cuuint64_t)(k64 * 64), (cuuint64_t)(I / 128), (cuuint64_t)(2 * a.experts)};
        const cuuint64_t ss[2] = {(cuuint64_t)(k64 * 512), (cuuint64_t)((I / 128) * k64 * 512)};
        const cuuint32_t sb[3] = {256u, 1u, 2u};
        if (!make_tmap(&tmSFB, a.b_sf, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, sd, ss, sb, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else {
        const cuuint64_t d[2] = {(cuuint64_t)kb, (cuuint64_t)(a.experts * a.N)};
        const cuuint64_t s[1] = {(cuuint64_t)kb};
        const cuuint32_t b[2] = {128u, 256u};
        if (!make_tmap(&tmB, a.b_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, d, s, b, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
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
    p.out_vec32 = (reinterpret_cast<uintptr_t>(a.out) % 32 == 0) && ((a.ldo * 2) % 32 == 0);
    p.n_tiles = swiglu ? (int32_t)(a.N / 256) : (int32_t)((a.N + 255) / 256);
    // persistent: at most one CTA per SM, never more CTAs than the largest possible tile count
    const int64_t max_tiles = ((a.m_capacity + 127) / 128) * p.n_tiles;
    const int64_t grid = std::min<int64_t>(max_tiles, a.sms);
    if (grid <= 0) return cudaSuccess;
    if (mx8) {
        if (a.epilogue == BSQ_EPI_BF16)
            k_gemm_fp4<BSQ_EPI_BF16, 1><<<(unsigned)grid, GmCfg<BSQ_EPI_BF16>::THREADS, GmCfg<BSQ_EPI_BF16>::SMEM_BYTES,
                                          st>>>(tmA, tmB, tmSFB, tmOut, p);
        else
            k_gemm_fp4<BSQ_EPI_F32, 1><<<(unsigned)grid, GmCfg<BSQ_EPI_F32>::THREADS, GmCfg<BSQ_EPI_F32>::SMEM_BYTES,
                                         st>>>(tmA, tmB, tmSFB, tmOut, p);
    } else if (swiglu)
        k_gemm_fp4<BSQ_EPI_SWIGLU_BF16><<<(unsigned)grid, GmCfg<BSQ_EPI_SWIGLU_BF16>::THREADS, GmCfg<BSQ_EPI_SWIGLU_BF16>::SMEM_BYTES, st>>>(
            tmA, tmB, tmSFB, tmOut, p);
    else if (a.epilogue == BSQ_EPI_BF16)
        k_gemm_fp4<BSQ_EPI_BF16><<<(unsigned)grid, GmCfg<BSQ_EPI_BF16>::THREADS, GmCfg<BSQ_EPI_BF16>::SMEM_BYTES, st>>>(tmA, tmB, tmSFB,
                                                                                                     tmOut, p);
    else
        k_gemm_fp4<BSQ_EPI_F32><<<(unsigned)grid, GmCfg<BSQ_EPI_F32>::THREADS, GmCfg<BSQ_EPI_F32>::SMEM_BYTES, st>>>(tmA, tmB, tmSFB,
                                                                                                   tmOut, p);
    return cudaGetLastError();
}

}  // namespace bsq
