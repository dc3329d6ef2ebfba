// ceiling.cu -- the block-scaled MMA ceiling of this GPU, measured: the rate at
// which the tensor cores retire back-to-back tcgen05.mma instructions of the
// forms the grouped GEMM issues, with operands already in shared memory and
// scale factors already in tensor memory (no copies, no epilogue).  This is
// the denominator of the GEMM's roofline fraction; the pages quote only
// nominal figures for it ("End-to-End 4-Bit Training", section "先说为什么难":
// the NVFP4 throughput of GB300).
//
// One CTA per SM (the shared-memory request keeps a second one off the SM),
// 128 threads.  FMT 0: kind::mxf4nvf4 scale_vec::4X, 128 x 256 x 64 per CTA
// per instruction; FMT 1: kind::mxf8f6f4 scale_vec::1X, 128 x 256 x 32.
// CG 2: clusters of two CTAs, one cta_group::2 MMA of 256 x 256 issued by the
// pair's first CTA (each CTA holds 128 rows of A and of B).  The issuing
// thread records clock64 from its first issue to the completion of the last
// MMA.  Every wait is bounded.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace bsq {
namespace {

constexpr uint32_t kCeilSpinLimit = 1u << 24;
constexpr int kCeilSmem = 120 * 1024;  // > half the SM's shared memory: one CTA per SM

BSQ_DEVICE bool ceil_wait(uint32_t bar)
{
    for (uint32_t i = 0; i < kCeilSpinLimit; ++i)
        if (mbar_try_wait(bar, 0u)) return true;
    return false;
}

template <int FMT, int CG>
__global__ void __launch_bounds__(128, 1) k_mma_ceiling(int32_t iters, unsigned long long* cycles, int32_t* dev_status)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t s_tmem;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;

    // operands: A [128 rows][128 B] at 0 and B [256 / CG rows][128 B] at 16 KB,
    // all zero codes (the MMA's duration does not depend on the values)
    constexpr int kBytes = 16384 + (256 / CG) * 128;
    for (int i = tid; i < kBytes / 16; i += 128) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const uint32_t b = smem_u32(&bar);
    if (tid == 0) {
        mbar_init(b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc<CG>(smem_u32(&s_tmem), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    {   // scale factors 1.0 in every byte of columns 256..287, all four lane quadrants
        const uint32_t one = FMT == 0 ? 0x38383838u : 0x7F7F7F7Fu;  // E4M3 1.0 / E8M0 2^0
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = one;
        const uint32_t quad = (uint32_t)warp << 21;  // lane 32 * warp, in bits 16..
        tc_st16(tmem + quad + 256, v);
        tc_st16(tmem + quad + 272, v);
        tc_st_wait();
    }
    tc_fence_before();
    if constexpr (CG == 2)
        cluster_sync();  // both CTAs' operands, scale factors and barriers are in place
    else
        __syncthreads();
    tc_fence_after();

    unsigned long long t0 = 0;
    if (rank == 0 && tid == 0) {
        const uint32_t sb = smem_u32(smem);
        const uint64_t ad = smem_desc(sb, 16, 1024, 2), bd = smem_desc(sb + 16384, 16, 1024, 2);
        const uint32_t idesc = FMT == 0 ? idesc_nvf4(256, 128 * CG) : idesc_mxf8(256, 0, 128 * CG);
        t0 = clock64();
        for (int i = 0; i < iters; ++i)  // the four K steps of a 128-byte stage, cycled
            tc_mma_bs<FMT, CG>(tmem, ad + 2 * (i & 3), bd + 2 * (i & 3), idesc, tmem + 256, tmem + 272,
                               i > 0 ? 1u : 0u);
        tc_commit<CG>(b);
    }
    bool ok = ceil_wait(b);
    if (rank == 0 && tid == 0) cycles[blockIdx.x] = ok ? clock64() - t0 : 0ull;
    if (!ok) {
        report(dev_status, BSQ_DEV_TIMEOUT);
        ceil_wait(b);  // tensor memory is freed only after the MMAs have completed
    }
    if (rank != 0 && tid == 0) cycles[blockIdx.x] = 0ull;
    tc_fence_before();
    if constexpr (CG == 2)
        cluster_sync();
    else
        __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc<CG>(tmem, 512);
    if constexpr (CG == 2) cluster_sync();
}

template <int FMT, int CG>
cudaError_t launch_one(int iters, unsigned long long* cycles, int32_t* dev_status, int ctas, cudaStream_t st)
{
    cudaError_t err = cudaFuncSetAttribute(k_mma_ceiling<FMT, CG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kCeilSmem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = kCeilSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_mma_ceiling<FMT, CG>, (int32_t)iters, cycles, dev_status);
}

}  // namespace

cudaError_t launch_mma_ceiling(int fmt, int cta_group, int iters, unsigned long long* cycles, int32_t* dev_status,
                               int ctas, cudaStream_t st)
{
    if (fmt == 0)
        return cta_group == 2 ? launch_one<0, 2>(iters, cycles, dev_status, ctas, st)
                              : launch_one<0, 1>(iters, cycles, dev_status, ctas, st);
    return cta_group == 2 ? launch_one<1, 2>(iters, cycles, dev_status, ctas, st)
                          : launch_one<1, 1>(iters, cycles, dev_status, ctas, st);
}

}  // namespace bsq
