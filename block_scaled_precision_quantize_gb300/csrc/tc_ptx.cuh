// tc_ptx.cuh -- inline-PTX wrappers for the 5th-generation tensor cores
// (tcgen05: MMA, tensor-memory allocation, copies and loads), the tensor-memory
// accelerator (cp.async.bulk / cp.async.bulk.tensor) and mbarriers, written
// from the public PTX ISA for sm_103a.  CG is the instruction's cta_group:
// 1 for one CTA, 2 for a pair of CTAs on neighbouring SMs (a cluster of two)
// that share one MMA: the pair's first CTA issues it, each CTA's shared memory
// holds its half of A's rows and of B's N rows, and each CTA's tensor memory
// receives its 128 rows of D.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace bsq {

BSQ_DEVICE uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ---------------------------------------------------------------- mbarrier
BSQ_DEVICE void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
BSQ_DEVICE void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
BSQ_DEVICE void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Arrive on a barrier of any CTA of the cluster (a shared::cluster address)
// with the default semantics (release at CTA scope).  Release at cluster scope
// would first wait for every earlier global store of the thread to become
// visible to the cluster, which costs the epilogue thousands of cycles per
// tile; the tensor-memory hand-off it signals is ordered by the tcgen05
// fences around it instead.
BSQ_DEVICE void mbar_arrive_cluster(uint32_t cluster_bar)
{
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
// Expect-tx on a barrier of any CTA of the cluster, counting one arrival.
BSQ_DEVICE void mbar_expect_tx_cluster(uint32_t cluster_bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_bar),
                 "r"(bytes)
                 : "memory");
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
// The same with acquire at cluster scope: for a barrier that the other CTA of
// a pair arrives on.
BSQ_DEVICE bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// ---------------------------------------------------------------- clusters
BSQ_DEVICE uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The same shared-memory offset in CTA `rank` of the cluster, as a
// shared::cluster address.
BSQ_DEVICE uint32_t mapa_shared(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
BSQ_DEVICE void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
// Tensor loads into this CTA's shared memory, completing on `bar`.  With
// CG = 2 (.cta_group::2) the barrier may be that of either CTA of the pair
// (a shared::cluster address).
template <int CG = 1>
BSQ_DEVICE void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar)
{
    if constexpr (CG == 2)
        asm volatile(
            "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
            "%3}], [%4];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
            : "memory");
    else
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
                dst),
            "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
            : "memory");
}
template <int CG = 1>
BSQ_DEVICE void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int x, int y, int z, uint32_t bar)
{
    if constexpr (CG == 2)
        asm volatile(
            "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
            "%3, %4}], [%5];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar)
            : "memory");
    else
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
            "[%5];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar)
            : "memory");
}
template <int CG = 1>
BSQ_DEVICE void tma_load_4d(uint32_t dst, const CUtensorMap* tm, int x, int y, int z, int w, uint32_t bar)
{
    if constexpr (CG == 2)
        asm volatile(
            "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
            "%3, %4, %5}], [%6];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
            : "memory");
    else
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
            "[%6];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
            : "memory");
}
// Untiled bulk copy global -> this CTA's shared memory (16-byte aligned
// addresses, size a multiple of 16), completing on `bar` (a shared::cluster
// address: this CTA's own barrier, or the pair's first CTA's).
BSQ_DEVICE void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// ---------------------------------------------------------------- tcgen05
BSQ_DEVICE void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
BSQ_DEVICE void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Allocation of `cols` tensor-memory columns (a power of two >= 32) by one
// whole warp; with CG = 2 one warp of each CTA of the pair allocates together.
// The base address is written to shared memory at dst_smem.
template <int CG = 1>
BSQ_DEVICE void tmem_alloc(uint32_t dst_smem, uint32_t cols)
{
    if constexpr (CG == 2) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
}
template <int CG = 1>
BSQ_DEVICE void tmem_dealloc(uint32_t taddr, uint32_t cols)
{
    if constexpr (CG == 2)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}

// Arrive on `bar` once every tcgen05 MMA and copy this thread issued before
// has completed.  With CG = 2 the arrival is multicast to the barrier at this
// offset in every CTA of `cta_mask`.
template <int CG = 1>
BSQ_DEVICE void tc_commit(uint32_t bar, uint16_t cta_mask = 3)
{
    if constexpr (CG == 2)
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                bar),
            "h"(cta_mask)
            : "memory");
    else
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

// One 512-byte scale-factor chunk (32 rows of 16 bytes in shared memory) into
// four tensor-memory columns, replicated in all four lane quadrants.  With
// CG = 2 (issued by the pair's first CTA) each CTA's chunk at this offset
// lands in its own tensor memory.
template <int CG = 1>
BSQ_DEVICE void tc_cp_sf(uint32_t taddr, uint64_t sdesc)
{
    if constexpr (CG == 2)
        asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
    else
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Block-scaled MMAs, D (tensor memory) [+]= A (smem) x B (smem)^T with scale
// factors in tensor memory.  FMT 0: kind::mxf4nvf4 scale_vec::4X (E2M1, E4M3
// scale per 16, K = 64); FMT 1: kind::mxf8f6f4 scale_vec::1X (E4M3, E8M0 scale
// per 32, K = 32).
template <int FMT, int CG = 1>
BSQ_DEVICE void tc_mma_bs(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                          uint32_t accumulate)
{
#define BSQ_MMA_ASM(CGS, KIND)                                                                                \
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"                                            \
                 "tcgen05.mma.cta_group::" CGS "." KIND " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),     \
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)                        \
                 : "memory")
    if constexpr (FMT == 0) {
        if constexpr (CG == 2)
            BSQ_MMA_ASM("2", "kind::mxf4nvf4.block_scale.scale_vec::4X");
        else
            BSQ_MMA_ASM("1", "kind::mxf4nvf4.block_scale.scale_vec::4X");
    } else {
        if constexpr (CG == 2)
            BSQ_MMA_ASM("2", "kind::mxf8f6f4.block_scale.scale_vec::1X");
        else
            BSQ_MMA_ASM("1", "kind::mxf8f6f4.block_scale.scale_vec::1X");
    }
#undef BSQ_MMA_ASM
}

// The same MMA with two barrier polls issued just before it in the same
// instruction stream: the tensor core's queue holds about one MMA, so a
// blocking barrier wait between MMAs leaves the tensor pipe idle for the
// wait's latency (~150 cycles), while polls issued ahead of an MMA and
// resolved after it cost nothing.  Returns bit 0 = phase `parity1` of `bar1`
// complete, bit 1 = phase `parity2` of `bar2` complete (non-blocking tests).
template <int FMT, int CG = 1>
BSQ_DEVICE uint32_t tc_mma_bs_poll2(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                    uint32_t sfb, uint32_t accumulate, uint32_t bar1, uint32_t parity1, uint32_t bar2,
                                    uint32_t parity2)
{
    uint32_t r;
#define BSQ_MMA_POLL_ASM(CGS, KIND)                                                                            \
    asm volatile("{\n\t.reg .pred p, q1, q2;\n\t.reg .b32 t1, t2;\n\t"                                         \
                 "mbarrier.test_wait.parity.shared::cta.b64 q1, [%8], %9;\n\t"                                \
                 "mbarrier.test_wait.parity.shared::cta.b64 q2, [%10], %11;\n\t"                              \
                 "setp.ne.b32 p, %5, 0;\n\t"                                                                  \
                 "tcgen05.mma.cta_group::" CGS "." KIND " [%1], %2, %3, %4, [%6], [%7], p;\n\t"                  \
                 "selp.u32 t1, 1, 0, q1;\n\t"                                                                 \
                 "selp.u32 t2, 2, 0, q2;\n\t"                                                                 \
                 "or.b32 %0, t1, t2;\n\t}"                                                                    \
                 : "=r"(r)                                                                                     \
                 : "r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb), "r"(bar1),  \
                   "r"(parity1), "r"(bar2), "r"(parity2)                                                        \
                 : "memory")
    if constexpr (FMT == 0) {
        if constexpr (CG == 2)
            BSQ_MMA_POLL_ASM("2", "kind::mxf4nvf4.block_scale.scale_vec::4X");
        else
            BSQ_MMA_POLL_ASM("1", "kind::mxf4nvf4.block_scale.scale_vec::4X");
    } else {
        if constexpr (CG == 2)
            BSQ_MMA_POLL_ASM("2", "kind::mxf8f6f4.block_scale.scale_vec::1X");
        else
            BSQ_MMA_POLL_ASM("1", "kind::mxf8f6f4.block_scale.scale_vec::1X");
    }
#undef BSQ_MMA_POLL_ASM
    return r;
}

// Instruction descriptors.  kind::mxf4nvf4: A and B are E2M1 (format 1),
// K-major, no negation, N >> 3 at bit 17, M >> 4 at bit 24 (128 for one CTA,
// 256 for a pair), scale type UE4M3 (bit 23 = 0), scale-factor ids 0, dense,
// K = 64.
__host__ __device__ constexpr uint32_t idesc_nvf4(uint32_t n, uint32_t m = 128)
{
    return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}
// kind::mxf8f6f4 with scale_vec::1X: A and B E4M3 (format 0), scale type
// UE8M0 (bit 23), K = 32.  Each tensor-memory scale column holds four E8M0
// bytes of a row, those of four consecutive 32-element blocks; the byte an
// MMA reads is its scale-factor id (B's at bits 4-5, A's at bits 29-30).
__host__ __device__ constexpr uint32_t idesc_mxf8(uint32_t n, uint32_t sf_id, uint32_t m = 128)
{
    return (sf_id << 4) | ((n >> 3) << 17) | (1u << 23) | ((m >> 4) << 24) | (sf_id << 29);
}

// 32 consecutive accumulator columns of this warp's 32 lanes, without waiting.
BSQ_DEVICE void tc_ld32_issue(uint32_t taddr, uint32_t r[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
// Wait for this thread's outstanding tcgen05.ld, then make every loaded
// register depend on the wait so no use can be scheduled before it.
template <int N>
BSQ_DEVICE void tc_ld_wait(uint32_t (&r)[N])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}
// Store 16 consecutive tensor-memory columns of this warp's 32 lanes.
BSQ_DEVICE void tc_st16(uint32_t taddr, const uint32_t* r)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
BSQ_DEVICE void tc_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- warp-issued forms
// The tcgen05 and TMA instructions take their descriptors, addresses and
// coordinates in warp-uniform registers.  Issued from a single active lane
// (inside `if (lane == 0)`), every operand must first be made uniform, which
// measured 2-3x slower MMA issue (280-420 cycles per 128-cycle MMA).  These
// forms are called by all 32 lanes of a converged warp with identical
// operands; one lane, chosen by elect.sync inside the instruction sequence,
// executes the instruction.  elect.sync picks the lowest active lane, so
// successive calls from a converged warp issue from the same lane, which
// tcgen05.commit needs (it tracks the issuing thread's own earlier MMAs and
// copies); the drains that guard the release of tensor memory do not rely on
// that (tc_commit_all).
#define BSQ_ELECT "{\n\t.reg .pred e_;\n\t.reg .b32 l_;\n\telect.sync l_|e_, 0xffffffff;\n\t"

template <int FMT, int CG = 1>
BSQ_DEVICE void tc_mma_bs_w(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                            uint32_t accumulate)
{
#define BSQ_MMA_W(CGS, KIND)                                                                                 \
    asm volatile(BSQ_ELECT ".reg .pred p_;\n\tsetp.ne.b32 p_, %4, 0;\n\t"                                     \
                 "@e_ tcgen05.mma.cta_group::" CGS "." KIND " [%0], %1, %2, %3, [%5], [%6], p_;\n\t}" ::"r"(d), \
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)                       \
                 : "memory")
    if constexpr (FMT == 0) {
        if constexpr (CG == 2)
            BSQ_MMA_W("2", "kind::mxf4nvf4.block_scale.scale_vec::4X");
        else
            BSQ_MMA_W("1", "kind::mxf4nvf4.block_scale.scale_vec::4X");
    } else {
        if constexpr (CG == 2)
            BSQ_MMA_W("2", "kind::mxf8f6f4.block_scale.scale_vec::1X");
        else
            BSQ_MMA_W("1", "kind::mxf8f6f4.block_scale.scale_vec::1X");
    }
#undef BSQ_MMA_W
}

// tc_mma_bs_w with two non-blocking barrier tests issued just before the MMA
// (by every lane): the tensor core's queue holds about one MMA, so a blocking
// barrier wait between MMAs leaves the pipe idle for the wait's latency, while
// tests issued ahead of an MMA and resolved after it cost nothing.  Returns
// bit 0 = phase `parity1` of `bar1` complete, bit 1 = phase `parity2` of `bar2`.
template <int FMT, int CG = 1>
BSQ_DEVICE uint32_t tc_mma_bs_poll2_w(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                      uint32_t sfb, uint32_t accumulate, uint32_t bar1, uint32_t parity1,
                                      uint32_t bar2, uint32_t parity2)
{
    uint32_t r;
#define BSQ_MMA_POLL_W(CGS, KIND)                                                                            \
    asm volatile(BSQ_ELECT ".reg .pred p_, q1_, q2_;\n\t.reg .b32 t1_, t2_;\n\t"                              \
                 "mbarrier.test_wait.parity.shared::cta.b64 q1_, [%8], %9;\n\t"                               \
                 "mbarrier.test_wait.parity.shared::cta.b64 q2_, [%10], %11;\n\t"                             \
                 "setp.ne.b32 p_, %5, 0;\n\t"                                                                 \
                 "@e_ tcgen05.mma.cta_group::" CGS "." KIND " [%1], %2, %3, %4, [%6], [%7], p_;\n\t"             \
                 "selp.u32 t1_, 1, 0, q1_;\n\t"                                                               \
                 "selp.u32 t2_, 2, 0, q2_;\n\t"                                                               \
                 "or.b32 %0, t1_, t2_;\n\t}"                                                                  \
                 : "=r"(r)                                                                                    \
                 : "r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb), "r"(bar1), \
                   "r"(parity1), "r"(bar2), "r"(parity2)                                                       \
                 : "memory")
    if constexpr (FMT == 0) {
        if constexpr (CG == 2)
            BSQ_MMA_POLL_W("2", "kind::mxf4nvf4.block_scale.scale_vec::4X");
        else
            BSQ_MMA_POLL_W("1", "kind::mxf4nvf4.block_scale.scale_vec::4X");
    } else {
        if constexpr (CG == 2)
            BSQ_MMA_POLL_W("2", "kind::mxf8f6f4.block_scale.scale_vec::1X");
        else
            BSQ_MMA_POLL_W("1", "kind::mxf8f6f4.block_scale.scale_vec::1X");
    }
#undef BSQ_MMA_POLL_W
    return r;
}

// tcgen05.commit from the elected lane (the one that issued the tracked MMAs
// or copies); CG 2 multicasts to the barrier at this offset in the CTAs of
// cta_mask.
template <int CG = 1>
BSQ_DEVICE void tc_commit_w(uint32_t bar, uint16_t cta_mask = 3)
{
    if constexpr (CG == 2)
        asm volatile(BSQ_ELECT "@e_ tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
                               "[%0], %1;\n\t}" ::"r"(bar),
                     "h"(cta_mask)
                     : "memory");
    else
        asm volatile(BSQ_ELECT "@e_ tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
                         bar)
                     : "memory");
}
// tcgen05.commit from every lane of the warp: the barrier (initialised with a
// count of 32) completes once the asynchronous tcgen05 work of whichever lane
// issued it has completed.  Guards the release of tensor memory.
template <int CG = 1>
BSQ_DEVICE void tc_commit_all(uint32_t bar, uint16_t cta_mask = 3)
{
    tc_commit<CG>(bar, cta_mask);
}

template <int CG = 1>
BSQ_DEVICE void tc_cp_sf_w(uint32_t taddr, uint64_t sdesc)
{
    if constexpr (CG == 2)
        asm volatile(BSQ_ELECT "@e_ tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr), "l"(sdesc)
                     : "memory");
    else
        asm volatile(BSQ_ELECT "@e_ tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr), "l"(sdesc)
                     : "memory");
}

BSQ_DEVICE void mbar_expect_tx_w(uint32_t bar, uint32_t bytes)
{
    asm volatile(BSQ_ELECT "@e_ mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes)
                 : "memory");
}

template <int CG = 1>
BSQ_DEVICE void tma_load_2d_w(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar)
{
    if constexpr (CG == 2)
        asm volatile(BSQ_ELECT "@e_ cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
                               "[%0], [%1, {%2, %3}], [%4];\n\t}" ::"r"(dst),
                     "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
                     : "memory");
    else
        asm volatile(BSQ_ELECT "@e_ cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
                               "{%2, %3}], [%4];\n\t}" ::"r"(dst),
                     "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
                     : "memory");
}
template <int CG = 1>
BSQ_DEVICE void tma_load_3d_w(uint32_t dst, const CUtensorMap* tm, int x, int y, int z, uint32_t bar)
{
    if constexpr (CG == 2)
        asm volatile(BSQ_ELECT "@e_ cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
                               "[%0], [%1, {%2, %3, %4}], [%5];\n\t}" ::"r"(dst),
                     "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar)
                     : "memory");
    else
        asm volatile(BSQ_ELECT "@e_ cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
                               "{%2, %3, %4}], [%5];\n\t}" ::"r"(dst),
                     "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar)
                     : "memory");
}
template <int CG = 1>
BSQ_DEVICE void tma_load_4d_w(uint32_t dst, const CUtensorMap* tm, int x, int y, int z, int w, uint32_t bar)
{
    if constexpr (CG == 2)
        asm volatile(BSQ_ELECT "@e_ cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
                               "[%0], [%1, {%2, %3, %4, %5}], [%6];\n\t}" ::"r"(dst),
                     "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
                     : "memory");
    else
        asm volatile(BSQ_ELECT "@e_ cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
                               "{%2, %3, %4, %5}], [%6];\n\t}" ::"r"(dst),
                     "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
                     : "memory");
}
BSQ_DEVICE void bulk_load_w(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile(BSQ_ELECT "@e_ cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}" ::"r"(
                     dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

}  // namespace bsq
