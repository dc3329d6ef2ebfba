/*
 * bsq_oracle.h -- plain, slow, single-threaded CPU oracle for block-scaled
 * NVFP4 / MXFP8 quantization and the block-scaled grouped expert GEMM.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, includes
 * or calls this code; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg do. It shares no source with the CUDA path.
 *
 * Conventions
 *  - bf16 inputs are passed as their raw 16-bit patterns (uint16_t).
 *  - NVFP4 codes: two E2M1 codes per byte, the element with the even K
 *    index in the low nibble.
 *  - NVFP4 scale factors (SF) are returned in the linear layout
 *    [rows][K/16] (one E4M3 byte per 16-element block along K).
 *  - MXFP8 codes are E4M3 bytes; MXFP8 SF are E8M0 bytes, one per 32
 *    elements along the reduction dimension.
 *  - "rn" below means one IEEE-754 binary32 operation rounded to nearest
 *    even; the file is compiled with -ffp-contract=off and without fast math
 *    so every float operation is exactly one rn step.
 */
#ifndef BSQ_ORACLE_H
#define BSQ_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element formats */
float    bsqo_e2m1_decode(uint32_t code);
uint32_t bsqo_e2m1_encode(float v);
uint32_t bsqo_e2m1_encode_sr(float v, uint32_t r16);
float    bsqo_e4m3_decode(uint32_t code);
uint32_t bsqo_e4m3_encode(float v);
uint32_t bsqo_e4m3_encode_sr(float v, uint32_t r16);
float    bsqo_e8m0_decode(uint32_t code);
void     bsqo_e2m1_encode_array(const float* v, int64_t n, uint8_t* out);
void     bsqo_e4m3_encode_array(const float* v, int64_t n, uint8_t* out);

/* counter-based random numbers */
void     bsqo_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
uint32_t bsqo_sr_bits16(uint64_t seed, uint32_t stream, uint64_t idx);

/* NVFP4 quantization */
void bsqo_nvfp4_quantize_rows(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx,
                              int four_six, uint8_t* codes, uint8_t* sf, float* t);
void bsqo_nvfp4_quantize_rows_given_t(const float* x, int64_t rows, int64_t K,
                                      const float* t, int four_six,
                                      uint8_t* codes, uint8_t* sf);
void bsqo_nvfp4_quantize_group(const uint16_t* x, int64_t groups, int64_t rows, int64_t K,
                               uint8_t* codes, uint8_t* sf, float* t);
void bsqo_nvfp4_block_candidate(const float* x16, float t, float mult,
                                uint8_t* code16, uint8_t* sf, float* sse);
void bsqo_nvfp4_dequantize(const uint8_t* codes, const uint8_t* sf, const float* t,
                           int64_t rows, int64_t K, float* out);
int64_t bsqo_sf_swizzled_offset(int64_t row, int64_t kblock, int64_t K);
void bsqo_sf_swizzle(const uint8_t* sf, int64_t rows, int64_t cols, uint8_t* out);

/* GEMM on exactly dequantized MXFP8 operands (fp64) */
void bsqo_gemm_mxfp8(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_t, int64_t M, int64_t K,
                     const uint8_t* b_codes, const uint8_t* b_sf, float b_t, int64_t N,
                     double* out, double* abs_out);

/* MXFP8 quantization */
void bsqo_mxfp8_quantize_rowcol(const uint16_t* x, int64_t rows, int64_t K, int64_t ldx,
                                uint8_t* row_codes, uint8_t* row_sf,
                                uint8_t* col_codes, uint8_t* col_sf);

/* 2-D NVFP4: one E4M3 scale per 16 x 16 tile, one FP32 scale per tensor */
void bsqo_nvfp4_quantize_2d(const uint16_t* x, int64_t rows, int64_t K,
                            uint8_t* codes, uint8_t* sf_tiles, float* t_out);

/* 32-point random Hadamard transform, and per-token NVFP4 of the transformed rows */
uint32_t bsqo_rht_signs(uint64_t seed);
void bsqo_rht32(const float* x, int64_t n, uint32_t signs, float* y);
void bsqo_nvfp4_quantize_rht(const uint16_t* x, int64_t rows, int64_t K, uint64_t seed,
                             uint8_t* codes, uint8_t* sf, float* t);

/* backward dequantize -> transpose -> requantize */
void bsqo_requant_transpose(const uint8_t* codes, const uint8_t* sf, const float* t,
                            int64_t rows, int64_t K, int sr, uint64_t seed,
                            uint8_t* nv_codes_T, uint8_t* nv_sf_T, float* nv_t_T,
                            uint8_t* mx_codes_T, uint8_t* mx_sf_T);

/* block-scaled GEMM on exactly dequantized operands (fp64) */
void bsqo_gemm_nvfp4(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_t,
                     int64_t M, int64_t K,
                     const uint8_t* b_codes, const uint8_t* b_sf, float b_t, int64_t N,
                     double* out, double* abs_out);
void bsqo_gemm_nvfp4_sampled(const uint8_t* a_codes, const uint8_t* a_sf, const float* a_t,
                             int64_t K,
                             const uint8_t* b_codes, const uint8_t* b_sf, const float* b_t,
                             const int64_t* a_rows, const int64_t* b_rows,
                             const int64_t* b_group, int64_t n_samples,
                             double* out, double* abs_out);

/* MoE expert forward pieces */
int64_t bsqo_route(const int32_t* topk_ids, int64_t T, int64_t k, int64_t E, int64_t pad,
                   int32_t* offsets, int32_t* slot_of, int32_t* row_src);
void bsqo_swiglu(const double* gate_up, int64_t rows, int64_t I, double* h);
void bsqo_combine(const uint16_t* out_rows, int64_t H, const int32_t* slot_of,
                  const float* topk_w, int64_t T, int64_t k, uint16_t* y);
uint16_t bsqo_f64_to_bf16(double v);
void bsqo_f64_to_bf16_array(const double* v, int64_t n, uint16_t* out);

#ifdef __cplusplus
}
#endif
#endif
