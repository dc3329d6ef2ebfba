// api.cu -- the C ABI (include/bsq.h): argument validation on the host,
// launches on the caller's stream.  No device memory is allocated here and
// no stream is synchronized.
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

using namespace bsq;

namespace {

constexpr int kMaxDevices = 64;

struct DevInfo {
    bool known;
    bool ok;
    int sms;
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

// The current device must be an sm_103 (GB300-class) part.
bsq_status current_device(int* sms)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BSQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return BSQ_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_dev_mutex);  // threads may share a device
    DevInfo& d = g_dev[dev];
    if (!d.known) {
        int major = 0, minor = 0, n = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return BSQ_ERR_CUDA;
        d.ok = (major == 10 && minor == 3);
        d.sms = n;
        d.known = true;
    }
    if (!d.ok) return BSQ_ERR_DEVICE;
    *sms = d.sms;
    return BSQ_OK;
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool a4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bsq_status launched()
{
    return cudaGetLastError() == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA;
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

thread_local void* const* t_stage_events = nullptr;

void stage_mark(int i, cudaStream_t st)
{
    if (t_stage_events) cudaEventRecord(static_cast<cudaEvent_t>(t_stage_events[i]), st);
}

int64_t moe_capacity(int64_t T, int64_t E, int64_t topk) { return ((T * topk + E * 127) + 127) / 128 * 128; }

}  // namespace

extern "C" {

const char* bsq_status_string(bsq_status s)
{
    switch (s) {
        case BSQ_OK: return "ok";
        case BSQ_ERR_NULL: return "null pointer";
        case BSQ_ERR_SHAPE: return "invalid shape";
        case BSQ_ERR_ALIGN: return "misaligned pointer or leading dimension";
        case BSQ_ERR_FLAGS: return "invalid flags";
        case BSQ_ERR_UNSUPPORTED: return "unsupported";
        case BSQ_ERR_CUDA: return "CUDA error";
        case BSQ_ERR_WORKSPACE: return "workspace missing or too small";
        case BSQ_ERR_DEVICE: return "current device is not sm_103";
    }
    return "unknown status";
}

int32_t bsq_version(void) { return 100; }

bsq_status bsq_check_status(const int32_t* dev_status, int32_t* status, bsq_stream_t stream)
{
    if (!dev_status || !status) return BSQ_ERR_NULL;
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, dev_status, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return BSQ_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return BSQ_ERR_CUDA;
    *status = v;
    return BSQ_OK;
}

bsq_status bsq_set_stage_events(void* const* events, int32_t n)
{
    if (events && n < 7) return BSQ_ERR_SHAPE;
    t_stage_events = events;
    return BSQ_OK;
}

bsq_status quantize_nvfp4_per_token(const void* x, int64_t rows, int64_t K, int64_t ldx, uint8_t* codes, uint8_t* sf,
                                    float* row_scale, uint32_t flags, int32_t* dev_status, bsq_stream_t stream)
{
    (void)dev_status;
    if (flags & ~(BSQ_SF_SWIZZLED | BSQ_FOUR_SIX)) return BSQ_ERR_FLAGS;
    if (rows < 0 || K <= 0 || K % 16 != 0 || K > 65536 || ldx < K || rows > (int64_t)1 << 31) return BSQ_ERR_SHAPE;
    if (rows == 0) return BSQ_OK;
    if (!x || !codes || !sf || !row_scale) return BSQ_ERR_NULL;
    if (!a16(x) || !a16(codes) || ldx % 8 != 0) return BSQ_ERR_ALIGN;
    int sms;
    bsq_status st = current_device(&sms);
    if (st != BSQ_OK) return st;
    launch_nvfp4_rows(static_cast<const uint16_t*>(x), rows, K, ldx, codes, sf, row_scale, nullptr, 1,
                      (flags & BSQ_FOUR_SIX) != 0, (flags & BSQ_SF_SWIZZLED) != 0, sms, true, stream);
    return launched();
}

bsq_status quantize_nvfp4_rht(const void* x, int64_t rows, int64_t K, int64_t ldx, uint64_t seed, uint8_t* codes,
                              uint8_t* sf, float* row_scale, uint32_t flags, int32_t* dev_status, bsq_stream_t stream)
{
    (void)dev_status;
    if (flags & ~BSQ_SF_SWIZZLED) return BSQ_ERR_FLAGS;
    if (rows < 0 || K <= 0 || K % 32 != 0 || K > 65536 || ldx < K || rows > (int64_t)1 << 31) return BSQ_ERR_SHAPE;
    if (rows == 0) return BSQ_OK;
    if (!x || !codes || !sf || !row_scale) return BSQ_ERR_NULL;
    if (!a16(x) || !a16(codes) || ldx % 8 != 0) return BSQ_ERR_ALIGN;
    int sms;
    bsq_status st = current_device(&sms);
    if (st != BSQ_OK) return st;
    launch_nvfp4_rht(static_cast<const uint16_t*>(x), rows, K, ldx, seed, codes, sf, row_scale,
                     (flags & BSQ_SF_SWIZZLED) != 0, sms, stream);
    return launched();
}

bsq_status quantize_nvfp4_2d(const void* x, int64_t rows, int64_t K, uint8_t* codes, uint8_t* sf_tiles,
                             uint8_t* codes_t, uint8_t* sf_tiles_t, float* tensor_scale, uint32_t flags,
                             int32_t* dev_status, bsq_stream_t stream)
{
    (void)dev_status;
    if (flags != 0) return BSQ_ERR_FLAGS;
    if (rows < 0 || K <= 0 || K % 16 != 0 || K > 65536 || rows % 16 != 0 || rows > (int64_t)1 << 31)
        return BSQ_ERR_SHAPE;
    if (rows == 0) return BSQ_OK;
    if (!x || !codes || !sf_tiles || !tensor_scale || (codes_t == nullptr) != (sf_tiles_t == nullptr))
        return BSQ_ERR_NULL;
    if (!a16(x) || !a16(codes) || (reinterpret_cast<uintptr_t>(codes_t) & 7u) ||
        (reinterpret_cast<uintptr_t>(tensor_scale) & 3u))
        return BSQ_ERR_ALIGN;
    int sms;
    bsq_status st = current_device(&sms);
    if (st != BSQ_OK) return st;
    if (launch_nvfp4_2d(static_cast<const uint16_t*>(x), rows, K, codes, sf_tiles, codes_t, sf_tiles_t, tensor_scale,
                        sms, stream) != cudaSuccess)
        return BSQ_ERR_CUDA;
    return launched();
}

bsq_status dequantize_nvfp4(const uint8_t* codes, const uint8_t* sf, const float* scale, int64_t rows, int64_t K,
                            int64_t group_rows, void* y, int64_t ldy, uint32_t flags, int32_t* dev_status,
                            bsq_stream_t stream)
{
    (void)dev_status;
    if (flags & ~BSQ_SF_SWIZZLED) return BSQ_ERR_FLAGS;
    if (rows < 0 || K <= 0 || K % 16 != 0 || K > 65536 || ldy < K || group_rows <= 0 || rows > (int64_t)1 << 31)
        return BSQ_ERR_SHAPE;
    if (rows == 0) return BSQ_OK;
    if (!codes || !sf || !scale || !y) return BSQ_ERR_NULL;
    if (!a16(codes) || !a16(y) || ldy % 8 != 0 || (reinterpret_cast<uintptr_t>(sf) & 3u)) return BSQ_ERR_ALIGN;
    int sms;
    bsq_status st = current_device(&sms);
    if (st != BSQ_OK) return st;
    launch_dequant_nvfp4(codes, sf, scale, rows, K, group_rows, static_cast<uint16_t*>(y), ldy,
                         (flags & BSQ_SF_SWIZZLED) != 0, sms, stream);
    return launched();
}

bsq_status quantize_nvfp4_per_expert(const void* w, int64_t experts, int64_t rows, int64_t K, uint8_t* codes,
                                     uint8_t* sf, float* expert_scale, uint32_t flags, int32_t* dev_status,
                                     bsq_stream_t stream)
{
    (void)dev_status;
    if (flags & ~BSQ_SF_SWIZZLED) return BSQ_ERR_FLAGS;
    if (experts < 0 || rows < 0 || K <= 0 || K % 16 != 0 || K > 65536) return BSQ_ERR_SHAPE;
    if ((flags & BSQ_SF_SWIZZLED) && rows % 128 != 0) return BSQ_ERR_SHAPE;
    if (experts * rows > (int64_t)1 << 31) return BSQ_ERR_SHAPE;
    if (experts == 0 || rows == 0) return BSQ_OK;
    if (!w || !codes || !sf || !expert_scale) return BSQ_ERR_NULL;
    if (!a16(w) || !a16(codes)) return BSQ_ERR_ALIGN;
    int sms;
    bsq_status st = current_device(&sms);
    if (st != BSQ_OK) return st;
    const uint16_t* x = static_cast<const uint16_t*>(w);
    if (cudaMemsetAsync(expert_scale, 0, (size_t)experts * sizeof(float), stream) != cudaSuccess) return BSQ_ERR_CUDA;
    launch_group_amax(x, experts * rows, K, rows, expert_scale, sms, stream);
    launch_nvfp4_rows(x, experts * rows, K, K, codes, sf, nullptr, expert_scale, rows, false,
                      (flags & BSQ_SF_SWIZZLED) != 0, sms, false, stream);
    launch_group_finalize(expert_scale, experts, stream);
    return launched();
}

bsq_status quantize_mxfp8_rowcol(const void* x, int64_t rows, int64_t K, int64_t ldx, uint8_t* row_codes,
                                 uint8_t* row_sf, uint8_t* col_codes, uint8_t* col_sf, uint32_t flags,
                                 int32_t* dev_status, bsq_stream_t stream)
{
    (void)dev_status;
    if (flags & ~BSQ_SF_SWIZZLED) return BSQ_ERR_FLAGS;
    if (rows < 0 || K <= 0 || rows % 32 != 0 || K % 32 != 0 || ldx < K || rows > (int64_t)1 << 31 ||
        K > (int64_t)1 << 31)
        return BSQ_ERR_SHAPE;
    if (rows == 0) return BSQ_OK;
    if (!x || (!row_codes && !col_codes)) return BSQ_ERR_NULL;
    if ((row_codes && !row_sf) || (col_codes && !col_sf)) return BSQ_ERR_NULL;
    if (!a16(x) || ldx % 8 != 0 || (row_codes && !a16(row_codes)) || (col_codes && !a16(col_codes)))
        return BSQ_ERR_ALIGN;
    if ((row_codes && !a4(row_sf)) || (col_codes && !a4(col_sf))) return BSQ_ERR_ALIGN;
    int sms;
    bsq_status st = current_device(&sms);
    if (st != BSQ_OK) return st;
    const bool swz = (flags & BSQ_SF_SWIZZLED) != 0;
    launch_mxfp8_rowcol(static_cast<const uint16_t*>(x), rows, K, ldx, row_codes, row_sf, col_codes, col_sf, swz,
                        stream);
    if (swz) {
        if (row_sf) launch_sf_pad_zero(row_sf, rows, K / 32, sms, stream);
        if (col_sf) launch_sf_pad_zero(col_sf, K, rows / 32, sms, stream);
    }
    return launched();
}

size_t bsq_requant_workspace_size(int64_t rows, int64_t K, int32_t nvfp4_target)
{
    if (!nvfp4_target || K <= 0 || rows <= 0) return 0;
    // the column maxima of |D| (K words, padded to 64)
    return align256((size_t)((K + 63) & ~(int64_t)63) * sizeof(float));
}

bsq_status requant_transpose_sr(const uint8_t* codes, const uint8_t* sf, const float* row_scale, int64_t rows,
                                int64_t K, uint8_t* nv_codes_T, uint8_t* nv_sf_T, float* nv_scale_T,
                                uint8_t* mx_codes_T, uint8_t* mx_sf_T, uint64_t seed, void* workspace,
                                size_t workspace_bytes, uint32_t flags, int32_t* dev_status, bsq_stream_t stream)
{
    (void)dev_status;
    if (flags & ~(BSQ_SF_SWIZZLED | BSQ_STOCHASTIC)) return BSQ_ERR_FLAGS;
    if (rows < 0 || K <= 0 || rows % 32 != 0 || K % 16 != 0 || rows > (int64_t)1 << 31 || K > (int64_t)1 << 31)
        return BSQ_ERR_SHAPE;
    if (rows == 0) return BSQ_OK;
    const bool nv = nv_codes_T || nv_sf_T || nv_scale_T;
    const bool mx = mx_codes_T || mx_sf_T;
    if (!codes || !sf || !row_scale) return BSQ_ERR_NULL;
    if (!nv && !mx) return BSQ_ERR_NULL;
    if (nv && (!nv_codes_T || !nv_sf_T || !nv_scale_T)) return BSQ_ERR_NULL;
    if (mx && (!mx_codes_T || !mx_sf_T)) return BSQ_ERR_NULL;
    if (!a16(codes) || (nv && !a16(nv_codes_T)) || (mx && !a16(mx_codes_T))) return BSQ_ERR_ALIGN;
    if (!a4(sf) || (nv && !a4(nv_sf_T)) || (mx && !a4(mx_sf_T))) return BSQ_ERR_ALIGN;
    const size_t need = bsq_requant_workspace_size(rows, K, nv ? 1 : 0);
    if (need && (!workspace || workspace_bytes < need)) return BSQ_ERR_WORKSPACE;
    int sms;
    bsq_status st = current_device(&sms);
    if (st != BSQ_OK) return st;
    const bool swz = (flags & BSQ_SF_SWIZZLED) != 0;
    if (launch_requant(codes, sf, row_scale, rows, K, static_cast<unsigned int*>(workspace), nv ? nv_codes_T : nullptr,
                       nv_sf_T, nv_scale_T, mx ? mx_codes_T : nullptr, mx_sf_T, seed, (flags & BSQ_STOCHASTIC) != 0,
                       swz, stream) != cudaSuccess)
        return BSQ_ERR_CUDA;
    if (swz) {
        if (nv) launch_sf_pad_zero(nv_sf_T, K, rows / 16, sms, stream);
        if (mx) launch_sf_pad_zero(mx_sf_T, K, rows / 32, sms, stream);
    }
    return launched();
}

bsq_status requant_transpose_sr_noalloc(const uint8_t* codes, const uint8_t* sf, const float* row_scale,
                                        int64_t rows, int64_t K, uint8_t* nv_codes_T, uint8_t* nv_sf_T,
                                        float* nv_scale_T, uint8_t* mx_codes_T, uint8_t* mx_sf_T, uint64_t seed,
                                        uint32_t flags, int32_t* dev_status, bsq_stream_t stream)
{
    (void)dev_status;
    if (flags & ~(BSQ_SF_SWIZZLED | BSQ_STOCHASTIC)) return BSQ_ERR_FLAGS;
    if (rows < 0 || K <= 0 || rows % 32 != 0 || K % 16 != 0 || rows > (int64_t)1 << 31) return BSQ_ERR_SHAPE;
    if (K > noalloc_requant_max_k()) return BSQ_ERR_SHAPE;  // beyond the library's fixed scratch array
    if (rows == 0) return BSQ_OK;
    const bool nv = nv_codes_T || nv_sf_T || nv_scale_T;
    const bool mx = mx_codes_T || mx_sf_T;
    if (!codes || !sf || !row_scale) return BSQ_ERR_NULL;
    if (!nv && !mx) return BSQ_ERR_NULL;
    if (nv && (!nv_codes_T || !nv_sf_T || !nv_scale_T)) return BSQ_ERR_NULL;
    if (mx && (!mx_codes_T || !mx_sf_T)) return BSQ_ERR_NULL;
    if (!a16(codes) || (nv && !a16(nv_codes_T)) || (mx && !a16(mx_codes_T))) return BSQ_ERR_ALIGN;
    if (!a4(sf) || (nv && !a4(nv_sf_T)) || (mx && !a4(mx_sf_T))) return BSQ_ERR_ALIGN;
    int sms;
    bsq_status st = current_device(&sms);
    if (st != BSQ_OK) return st;
    const bool swz = (flags & BSQ_SF_SWIZZLED) != 0;
    if (launch_requant_noalloc(codes, sf, row_scale, rows, K, nv ? nv_codes_T : nullptr, nv_sf_T, nv_scale_T,
                               mx ? mx_codes_T : nullptr, mx_sf_T, seed, (flags & BSQ_STOCHASTIC) != 0, swz,
                               stream) != cudaSuccess)
        return BSQ_ERR_CUDA;
    if (swz) {
        if (nv) launch_sf_pad_zero(nv_sf_T, K, rows / 16, sms, stream);
        if (mx) launch_sf_pad_zero(mx_sf_T, K, rows / 32, sms, stream);
    }
    return launched();
}

bsq_status grouped_expert_gemm_mxfp8(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_scale,
                                     const int32_t* offsets, int64_t experts, int64_t m_capacity, int64_t K, int64_t N,
                                     const uint8_t* b_codes, const uint8_t* b_sf, const float* b_scale,
                                     int32_t epilogue, void* out, int64_t ldo, uint32_t flags, int32_t* dev_status,
                                     bsq_stream_t stream)
{
    if (flags != 0 && flags != BSQ_SF_SWIZZLED) return BSQ_ERR_FLAGS;
    if (epilogue != BSQ_EPI_F32 && epilogue != BSQ_EPI_BF16) return BSQ_ERR_FLAGS;
    if (experts <= 0 || m_capacity < 0 || K <= 0 || N <= 0 || K % 128 != 0 || N % 128 != 0) return BSQ_ERR_SHAPE;
    if (ldo < N) return BSQ_ERR_SHAPE;
    if (m_capacity > ((int64_t)1 << 31) - 256 || experts * N > ((int64_t)1 << 31) - 256 || K > ((int64_t)1 << 20))
        return BSQ_ERR_SHAPE;
    if (m_capacity == 0) return BSQ_OK;
    if (!a_codes || !a_sf || !a_scale || !offsets || !b_codes || !b_sf || !b_scale || !out) return BSQ_ERR_NULL;
    const int64_t esz = epilogue == BSQ_EPI_F32 ? 4 : 2;
    if (!a16(a_codes) || !a16(b_codes) || !a16(a_sf) || !a16(b_sf) || !a16(out) || (ldo * esz) % 16 != 0)
        return BSQ_ERR_ALIGN;
    int sms;
    bsq_status st = current_device(&sms);
    if (st != BSQ_OK) return st;
    GemmArgs g;
    g.a_codes = a_codes;
    g.a_sf = a_sf;
    g.a_scale = a_scale;
    g.offsets = offsets;
    g.experts = experts;
    g.m_capacity = m_capacity;
    g.K = K;
    g.N = N;
    g.b_codes = b_codes;
    g.b_sf = b_sf;
    g.b_scale = b_scale;
    g.epilogue = epilogue;
    g.out = out;
    g.ldo = ldo;
    g.dev_status = dev_status;
    g.sms = sms;
    g.fmt = 1;
    return launch_gemm_fp4(g, stream) == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA;
}

bsq_status grouped_expert_gemm_fp4(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_scale,
                                   const int32_t* offsets, int64_t experts, int64_t m_capacity, int64_t K, int64_t N,
                                   const uint8_t* b_codes, const uint8_t* b_sf, const float* b_scale,
                                   int32_t epilogue, void* out, int64_t ldo, uint32_t flags, int32_t* dev_status,
                                   bsq_stream_t stream)
{
    if (flags != 0 && flags != BSQ_SF_SWIZZLED) return BSQ_ERR_FLAGS;
    if (epilogue != BSQ_EPI_F32 && epilogue != BSQ_EPI_BF16 && epilogue != BSQ_EPI_SWIGLU_BF16) return BSQ_ERR_FLAGS;
    if (experts <= 0 || m_capacity < 0 || K <= 0 || N <= 0 || K % 64 != 0 || N % 128 != 0) return BSQ_ERR_SHAPE;
    if (epilogue == BSQ_EPI_SWIGLU_BF16 && N % 256 != 0) return BSQ_ERR_SHAPE;
    const int64_t ncols = epilogue == BSQ_EPI_SWIGLU_BF16 ? N / 2 : N;
    if (ldo < ncols) return BSQ_ERR_SHAPE;
    if (m_capacity > ((int64_t)1 << 31) - 256 || experts * N > ((int64_t)1 << 31) - 256 || K > ((int64_t)1 << 20))
        return BSQ_ERR_SHAPE;
    if (m_capacity == 0) return BSQ_OK;
    if (!a_codes || !a_sf || !a_scale || !offsets || !b_codes || !b_sf || !b_scale || !out) return BSQ_ERR_NULL;
    const int64_t esz = epilogue == BSQ_EPI_F32 ? 4 : 2;
    if (!a16(a_codes) || !a16(b_codes) || !a16(a_sf) || !a16(b_sf) || !a16(out) || (ldo * esz) % 16 != 0)
        return BSQ_ERR_ALIGN;
    int sms;
    bsq_status st = current_device(&sms);
    if (st != BSQ_OK) return st;
    GemmArgs g;
    g.a_codes = a_codes;
    g.a_sf = a_sf;
    g.a_scale = a_scale;
    g.offsets = offsets;
    g.experts = experts;
    g.m_capacity = m_capacity;
    g.K = K;
    g.N = N;
    g.b_codes = b_codes;
    g.b_sf = b_sf;
    g.b_scale = b_scale;
    g.epilogue = epilogue;
    g.out = out;
    g.ldo = ldo;
    g.dev_status = dev_status;
    g.sms = sms;
    return launch_gemm_fp4(g, stream) == cudaSuccess ? BSQ_OK : BSQ_ERR_CUDA;
}

bsq_status bsq_moe_workspace_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk, bsq_moe_layout* L)
{
    if (!L) return BSQ_ERR_NULL;
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || topk <= 0 || topk > 32) return BSQ_ERR_SHAPE;
    std::memset(L, 0, sizeof(*L));
    const int64_t cap = moe_capacity(T, E, topk);
    const int64_t nchunks = (T * topk + 511) / 512;  // routing chunk of 512 pairs
    size_t o = 0;
    // each sub-buffer starts 256-byte aligned and is followed by at least 256
    // unused bytes, a guard band that tests fill with a canary and check
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align256(o + bytes) + 256;
        return at;
    };
    L->capacity = cap;
    L->offsets = take((size_t)(E + 1) * 4);
    L->counts = take((size_t)E * 4);
    L->slot_of = take((size_t)(T * topk) * 4);
    L->row_src = take((size_t)cap * 4);
    L->xq_codes = take((size_t)cap * (H / 2));
    L->xq_sf = take((size_t)cap * ((H / 16 + 3) / 4 * 4));
    L->xq_scale = take((size_t)cap * 4);
    L->h = take((size_t)cap * I * 2);
    L->hq_codes = take((size_t)cap * (I / 2));
    L->hq_sf = take((size_t)cap * ((I / 16 + 3) / 4 * 4));
    L->hq_scale = take((size_t)cap * 4);
    L->out = take((size_t)cap * H * 2);
    L->scan = take(((size_t)std::max<int64_t>(nchunks, 1) * E + 1) * 4);  // histograms + ticket
    L->h_scratch = take((size_t)2 * BSQ_MOE_MAX_CTAS * 128 * I * 2);  // two units per CTA
    L->total = o;
    return BSQ_OK;
}

size_t bsq_moe_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk)
{
    bsq_moe_layout L;
    return bsq_moe_workspace_layout(T, H, I, E, topk, &L) == BSQ_OK ? L.total : 0;
}

bsq_status moe_expert_forward(const void* x, int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk,
                              const int32_t* topk_ids, const float* topk_weights, const uint8_t* wgu_codes,
                              const uint8_t* wgu_sf, const float* wgu_scale, const uint8_t* wd_codes,
                              const uint8_t* wd_sf, const float* wd_scale, void* y, void* workspace,
                              size_t workspace_bytes, uint32_t flags, int32_t* dev_status, bsq_stream_t stream)
{
    if (flags & ~(BSQ_FOUR_SIX | BSQ_MOE_FUSED_H | BSQ_MOE_KEEP_H)) return BSQ_ERR_FLAGS;
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || topk <= 0 || topk > 32 || E > 4096) return BSQ_ERR_SHAPE;
    if (H % 128 != 0 || H > 8192 || I % 128 != 0 || I > 8192) return BSQ_ERR_SHAPE;
    if (T * topk > ((int64_t)1 << 30)) return BSQ_ERR_SHAPE;
    if (T == 0) return BSQ_OK;
    if (!x || !topk_ids || !topk_weights || !wgu_codes || !wgu_sf || !wgu_scale || !wd_codes || !wd_sf ||
        !wd_scale || !y)
        return BSQ_ERR_NULL;
    if (!a16(x) || !a16(y) || !a16(wgu_codes) || !a16(wd_codes) || !a16(wgu_sf) || !a16(wd_sf) || !a16(workspace))
        return BSQ_ERR_ALIGN;
    bsq_moe_layout L;
    bsq_status st = bsq_moe_workspace_layout(T, H, I, E, topk, &L);
    if (st != BSQ_OK) return st;
    if (!workspace || workspace_bytes < L.total) return BSQ_ERR_WORKSPACE;
    int sms;
    st = current_device(&sms);
    if (st != BSQ_OK) return st;
    if ((flags & BSQ_MOE_FUSED_H) && gemm_fp4_ctas(E, L.capacity, (2 * I) / 256, sms) > BSQ_MOE_MAX_CTAS)
        return BSQ_ERR_UNSUPPORTED;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    auto I32 = [&](size_t off) { return reinterpret_cast<int32_t*>(ws + off); };
    auto F32 = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
    const bool f46 = (flags & BSQ_FOUR_SIX) != 0;
    const int64_t cap = L.capacity;

    stage_mark(0, stream);
    launch_route(topk_ids, T, (int32_t)topk, (int32_t)E, I32(L.scan), I32(L.counts), I32(L.offsets), I32(L.slot_of),
                 I32(L.row_src), cap, dev_status, stream);
    stage_mark(1, stream);
    launch_quant_scatter(static_cast<const uint16_t*>(x), T, H, (int32_t)topk, I32(L.slot_of), I32(L.offsets),
                         I32(L.counts), (int32_t)E, ws + L.xq_codes, ws + L.xq_sf, F32(L.xq_scale), I32(L.row_src), cap, f46,
                         sms, stream);
    if (cudaGetLastError() != cudaSuccess) return BSQ_ERR_CUDA;
    stage_mark(2, stream);

    GemmArgs g1;
    g1.a_codes = ws + L.xq_codes;
    g1.a_sf = ws + L.xq_sf;
    g1.a_scale = F32(L.xq_scale);
    g1.offsets = I32(L.offsets);
    g1.experts = E;
    g1.m_capacity = cap;
    g1.K = H;
    g1.N = 2 * I;
    g1.b_codes = wgu_codes;
    g1.b_sf = wgu_sf;
    g1.b_scale = wgu_scale;
    g1.out = ws + L.h;
    g1.ldo = I;
    g1.dev_status = dev_status;
    g1.sms = sms;
    if (flags & BSQ_MOE_FUSED_H) {
        // SwiGLU with the per-token NVFP4 quantization of h fused in
        g1.epilogue = f46 ? GM_EPI_SWIGLU_Q46 : GM_EPI_SWIGLU_Q;
        g1.q_codes = ws + L.hq_codes;
        g1.q_sf = ws + L.hq_sf;
        g1.q_scale = F32(L.hq_scale);
        g1.h_scratch = reinterpret_cast<uint16_t*>(ws + L.h_scratch);
        g1.keep_h = (flags & BSQ_MOE_KEEP_H) != 0;
        if (launch_gemm_fp4(g1, stream) != cudaSuccess) return BSQ_ERR_CUDA;
        stage_mark(3, stream);
        stage_mark(4, stream);
    } else {
        // SwiGLU -> bf16 h, then the per-token quantizer over h
        g1.epilogue = BSQ_EPI_SWIGLU_BF16;
        if (launch_gemm_fp4(g1, stream) != cudaSuccess) return BSQ_ERR_CUDA;
        stage_mark(3, stream);
        launch_nvfp4_rows(reinterpret_cast<const uint16_t*>(ws + L.h), cap, I, I, ws + L.hq_codes, ws + L.hq_sf,
                          F32(L.hq_scale), nullptr, 1, f46, true, sms, true, stream);
        stage_mark(4, stream);
    }

    GemmArgs g2 = g1;
    g2.q_codes = g2.q_sf = nullptr;
    g2.q_scale = nullptr;
    g2.h_scratch = nullptr;
    g2.keep_h = false;
    g2.a_codes = ws + L.hq_codes;
    g2.a_sf = ws + L.hq_sf;
    g2.a_scale = F32(L.hq_scale);
    g2.K = I;
    g2.N = H;
    g2.b_codes = wd_codes;
    g2.b_sf = wd_sf;
    g2.b_scale = wd_scale;
    g2.epilogue = BSQ_EPI_BF16;
    g2.out = ws + L.out;
    g2.ldo = H;
    if (launch_gemm_fp4(g2, stream) != cudaSuccess) return BSQ_ERR_CUDA;
    stage_mark(5, stream);

    launch_combine(reinterpret_cast<const uint16_t*>(ws + L.out), T, H, (int32_t)topk, I32(L.slot_of), topk_weights,
                   static_cast<uint16_t*>(y), sms, stream);
    stage_mark(6, stream);
    return launched();
}

bsq_status bsq_mma_ceiling(int32_t fmt, int32_t cta_group, int32_t iters, uint64_t* cycles, int32_t* ctas,
                           int32_t* dev_status, bsq_stream_t stream)
{
    if ((fmt != 0 && fmt != 1) || (cta_group != 1 && cta_group != 2)) return BSQ_ERR_FLAGS;
    if (iters <= 0 || iters > 65536) return BSQ_ERR_SHAPE;
    if (!cycles || !ctas) return BSQ_ERR_NULL;
    int sms;
    bsq_status st = current_device(&sms);
    if (st != BSQ_OK) return st;
    const int n = sms / cta_group * cta_group;
    *ctas = n;
    if (launch_mma_ceiling(fmt, cta_group, iters, reinterpret_cast<unsigned long long*>(cycles), dev_status, n,
                           stream) != cudaSuccess)
        return BSQ_ERR_CUDA;
    return launched();
}

bsq_status bsq_sf_swizzle(const uint8_t* sf_linear, int64_t rows, int64_t cols, uint8_t* sf_swizzled,
                          bsq_stream_t stream)
{
    if (rows < 0 || cols <= 0) return BSQ_ERR_SHAPE;
    if (rows == 0) return BSQ_OK;
    if (!sf_linear || !sf_swizzled) return BSQ_ERR_NULL;
    int sms;
    bsq_status st = current_device(&sms);
    if (st != BSQ_OK) return st;
    launch_sf_swizzle(sf_linear, rows, cols, sf_swizzled, 0, sms, stream);
    return launched();
}

bsq_status bsq_sf_unswizzle(const uint8_t* sf_swizzled, int64_t rows, int64_t cols, uint8_t* sf_linear,
                            bsq_stream_t stream)
{
    if (rows < 0 || cols <= 0) return BSQ_ERR_SHAPE;
    if (rows == 0) return BSQ_OK;
    if (!sf_linear || !sf_swizzled) return BSQ_ERR_NULL;
    int sms;
    bsq_status st = current_device(&sms);
    if (st != BSQ_OK) return st;
    launch_sf_swizzle(sf_swizzled, rows, cols, sf_linear, 1, sms, stream);
    return launched();
}

bsq_status bsq_format_probe(int32_t kind, const float* in, const uint32_t* rbits, void* out, int64_t n,
                            bsq_stream_t stream)
{
    if (kind < 0 || kind > 5) return BSQ_ERR_FLAGS;
    if (n < 0) return BSQ_ERR_SHAPE;
    if (n == 0) return BSQ_OK;
    if (!in || !out || ((kind == 2 || kind == 3) && !rbits)) return BSQ_ERR_NULL;
    int sms;
    bsq_status st = current_device(&sms);
    if (st != BSQ_OK) return st;
    launch_format_probe(kind, in, rbits, out, n, sms, stream);
    return launched();
}

bsq_status bsq_philox_bits16(uint64_t seed, uint32_t stream_id, uint64_t idx0, int64_t n, uint16_t* out,
                             bsq_stream_t stream)
{
    if (n < 0) return BSQ_ERR_SHAPE;
    if (n == 0) return BSQ_OK;
    if (!out) return BSQ_ERR_NULL;
    int sms;
    bsq_status st = current_device(&sms);
    if (st != BSQ_OK) return st;
    launch_philox_bits16(seed, stream_id, idx0, n, out, sms, stream);
    return launched();
}

}  // extern "C"
