// kernels.h -- launchers of the device kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bsq {

void launch_nvfp4_rows(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx, uint8_t* codes, uint8_t* sf,
                       float* row_scale, const float* group_amax, int64_t rows_per_group, bool four_six, bool swz,
                       int sms, bool pdl, cudaStream_t st);
void launch_group_amax(const uint16_t* x, int64_t rows, int64_t K, int64_t rows_per_group, float* group_amax,
                       int sms, cudaStream_t st);
void launch_group_finalize(float* scale, int64_t groups, cudaStream_t st);
void launch_nvfp4_rht(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx, uint64_t seed, uint8_t* codes,
                      uint8_t* sf, float* row_scale, bool swz, int sms, cudaStream_t st);
cudaError_t launch_nvfp4_2d(const uint16_t* x, int64_t rows, int64_t K, uint8_t* codes, uint8_t* sf,
                            uint8_t* codes_t, uint8_t* sf_t, float* tscale, int sms, cudaStream_t st);
void launch_dequant_nvfp4(const uint8_t* codes, const uint8_t* sf, const float* scale, int64_t rows, int64_t K,
                          int64_t group_rows, uint16_t* y, int64_t ldy, bool swizzled, int sms, cudaStream_t st);
void launch_mxfp8_rowcol(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx, uint8_t* rc, uint8_t* rs,
                         uint8_t* cc, uint8_t* cs, bool swz, cudaStream_t st);
void launch_sf_pad_zero(uint8_t* sf, int64_t rows, int64_t cols, int sms, cudaStream_t st);
cudaError_t launch_requant(const uint8_t* codes, const uint8_t* sf, const float* row_scale, int64_t rows, int64_t K,
                           unsigned int* colmax, uint8_t* nvc, uint8_t* nvs, float* nvt, uint8_t* mxc, uint8_t* mxs,
                           uint64_t seed, bool sr, bool swz, cudaStream_t st);
int64_t noalloc_requant_max_k();
cudaError_t launch_requant_noalloc(const uint8_t* codes, const uint8_t* sf, const float* row_scale, int64_t rows,
                                   int64_t K, uint8_t* nvc, uint8_t* nvs, float* nvt, uint8_t* mxc, uint8_t* mxs,
                                   uint64_t seed, bool sr, bool swz, cudaStream_t st);
void launch_sf_swizzle(const uint8_t* in, int64_t rows, int64_t cols, uint8_t* out, int dir, int sms,
                       cudaStream_t st);
void launch_format_probe(int kind, const float* in, const uint32_t* rbits, void* out, int64_t n, int sms,
                         cudaStream_t st);
void launch_philox_bits16(uint64_t seed, uint32_t stream, uint64_t idx0, int64_t n, uint16_t* out, int sms,
                          cudaStream_t st);

struct GemmArgs {
    const uint8_t* a_codes;
    const uint8_t* a_sf;
    const float* a_scale;
    const int32_t* offsets;
    int64_t experts;
    int64_t m_capacity;
    int64_t K;
    int64_t N;
    const uint8_t* b_codes;
    const uint8_t* b_sf;
    const float* b_scale;
    int32_t epilogue;
    void* out;
    int64_t ldo;
    int32_t* dev_status;
    int sms;  // SMs of the current device (persistent grid size)
    int fmt = 0;  // 0: NVFP4 operands, 1: MXFP8 operands
    // the fused SwiGLU + NVFP4-of-h epilogue (GM_EPI_SWIGLU_Q / _Q46): the
    // quantized h, a scratch of 128 rows x N/2 bf16 per CTA, and whether h is
    // also kept in full in `out` (for staged checks) instead of the scratch
    uint8_t* q_codes = nullptr;
    uint8_t* q_sf = nullptr;
    float* q_scale = nullptr;
    uint16_t* h_scratch = nullptr;
    bool keep_h = false;
};
// Internal epilogue kinds (not part of the C ABI): SwiGLU with the per-token
// NVFP4 quantization of h fused in, without / with the 4/6 block-scale choice.
constexpr int GM_EPI_SWIGLU_Q = 8;
constexpr int GM_EPI_SWIGLU_Q46 = 9;
// The CTAs the grouped GEMM launches for a problem on `sms` SMs (the fused
// epilogue's scratch holds 128 rows of h per CTA).
int64_t gemm_fp4_ctas(int64_t experts, int64_t m_capacity, int64_t n_tiles, int sms);
cudaError_t launch_gemm_fp4(const GemmArgs& a, cudaStream_t st);
cudaError_t launch_mma_ceiling(int fmt, int cta_group, int iters, unsigned long long* cycles, int32_t* dev_status,
                               int ctas, cudaStream_t st);

void launch_route(const int32_t* ids, int64_t T, int32_t topk, int32_t E, int32_t* hist, int32_t* counts,
                  int32_t* offsets, int32_t* slot_of, int32_t* row_src, int64_t capacity, int32_t* dev_status,
                  cudaStream_t st);
void launch_quant_scatter(const uint16_t* x, int64_t T, int64_t H, int32_t topk, const int32_t* slot_of,
                          const int32_t* offsets, const int32_t* counts, int32_t E, uint8_t* codes, uint8_t* sf,
                          float* scale, int32_t* row_src, int64_t cap, bool four_six, int sms, cudaStream_t st);
void launch_combine(const uint16_t* out, int64_t T, int64_t H, int32_t topk, const int32_t* slot_of, const float* w,
                    uint16_t* y, int sms, cudaStream_t st);

}  // namespace bsq
