/*
 * bsq.h -- C ABI of the block-scaled quantization hot path for MoE experts on
 * GB300 (sm_103a): per-token NVFP4 and MXFP8 quantizers, the backward
 * dequantize -> transpose -> requantize step with stochastic rounding, and a
 * block-scaled grouped expert GEMM on the 5th-generation tensor cores, composed
 * into an MoE expert forward.
 *
 * Formats (as the pages state them):
 *  - NVFP4: E2M1 elements (magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6), one E4M3
 *    block scale per 16 consecutive values along the reduction dimension K, and
 *    one FP32 second-level scale ("Miles Blackwell RL ..." (remio.ai), section
 *    "Il supporto Miles Blackwell ora copre l'intero ciclo RL"; "End-to-End
 *    4-Bit Training" summary (nopree.com), section "先说为什么难").  The FP32
 *    scale is per token for activations and per expert for weights ("4ビットの
 *    教訓" (hackernews.jp), section "ベースラインレシピ").
 *  - MXFP8: E4M3 elements, one E8M0 scale per 32 consecutive values ("LMSYS
 *    Drops Miles ..." (alphasignal.ai), section "Recipe 1: End-to-end MXFP8").
 *
 * Memory and ownership.  Every tensor pointer is a DEVICE pointer (CUDA global
 * memory) owned by the caller; the library never allocates device memory,
 * never frees it and never synchronizes a stream.  All work is enqueued on
 * `stream` (a cudaStream_t; NULL = the legacy default stream) in call order.
 * Pointers must be 16-byte aligned and leading dimensions must keep every row
 * 16-byte aligned unless stated otherwise.
 *
 * Layouts.
 *  - bf16 / fp32 matrices are row-major with a leading dimension in elements.
 *  - NVFP4 codes: [rows][K/2] bytes, two E2M1 codes per byte, the element with
 *    the even K index in the low nibble.
 *  - Scale factors (SF), BSQ_SF_LINEAR: [rows][K/16] (NVFP4) or [rows][K/32]
 *    (MXFP8) bytes, row-major.
 *  - SF, BSQ_SF_SWIZZLED (the layout the block-scaled tensor-core MMA copies
 *    into tensor memory): the SF matrix is cut into tiles of 128 rows x 4 SF
 *    columns, stored tile-row major, 512 bytes per tile; SF (r, c) sits at
 *    ((r/128) * ceil(C/4) + c/4) * 512 + (r%32) * 16 + ((r%128)/32) * 4 + c%4,
 *    C = number of SF columns.  Buffers hold ceil(rows/128)*128 x
 *    ceil(C/4)*4 bytes; padding bytes are written as 0.
 *
 * Errors.  Every call returns a bsq_status.  Argument errors detectable on the
 * host (NULL pointers, shapes, alignment, flags, workspace size) are reported
 * before anything is enqueued.  BSQ_ERR_CUDA reports a launch failure.
 * Asynchronous device-side problems (a bounded wait that expired, an
 * out-of-range expert id or offset) are written to the optional caller-owned
 * device word `dev_status` (first error wins; the caller zeroes it); the
 * kernel that detects one skips the affected work and returns normally.
 * Inputs must be finite; SF bytes 0x7F/0xFF (E4M3 NaN) are outside the
 * contract.
 */
#ifndef BSQ_H
#define BSQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* bsq_stream_t; /* same type as cudaStream_t */

typedef enum {
    BSQ_OK = 0,
    BSQ_ERR_NULL = 1,        /* a required pointer is NULL */
    BSQ_ERR_SHAPE = 2,       /* a size is negative, too large or not a required multiple */
    BSQ_ERR_ALIGN = 3,       /* a pointer or leading dimension breaks 16-byte alignment */
    BSQ_ERR_FLAGS = 4,       /* unknown or contradictory flag bits */
    BSQ_ERR_UNSUPPORTED = 5, /* valid request this build does not implement */
    BSQ_ERR_CUDA = 6,        /* a CUDA runtime/driver call or a launch failed */
    BSQ_ERR_WORKSPACE = 7,   /* workspace NULL or smaller than required */
    BSQ_ERR_DEVICE = 8       /* no sm_103-class device is current */
} bsq_status;

/* Values written to dev_status by the kernels. */
#define BSQ_DEV_OK 0
#define BSQ_DEV_TIMEOUT 1       /* a bounded pipeline wait expired; the tile was skipped */
#define BSQ_DEV_BAD_OFFSETS 2   /* expert offsets not ascending multiples of 128 within capacity */
#define BSQ_DEV_BAD_EXPERT 3    /* a routed expert id outside [0, E) */

/* flags */
#define BSQ_SF_LINEAR 0u
#define BSQ_SF_SWIZZLED (1u << 0)   /* scale factors in the tensor-core tile layout */
#define BSQ_FOUR_SIX (1u << 1)      /* NVFP4 "4/6" block-scale choice (activations only) */
#define BSQ_STOCHASTIC (1u << 2)    /* stochastic rounding of element codes (requant) */
#define BSQ_MOE_FUSED_H (1u << 3)   /* moe_expert_forward: quantize h inside GEMM1's epilogue */
#define BSQ_MOE_KEEP_H (1u << 4)    /* with BSQ_MOE_FUSED_H: also keep the bf16 SwiGLU output h */

/* GEMM epilogues */
#define BSQ_EPI_F32 0         /* out fp32 [M][N] = acc * a_scale[row] * b_scale[expert] */
#define BSQ_EPI_BF16 1        /* out bf16 [M][N], same values rounded to nearest even */
#define BSQ_EPI_SWIGLU_BF16 2 /* out bf16 [M][N/2] = silu(y[:, :N/2]) * y[:, N/2:] */

const char* bsq_status_string(bsq_status s);
int32_t bsq_version(void);

/* bsq_check_status: reads a dev_status word back to the host.  It copies the
 * device int32 at dev_status into *status on `stream`, after the work already
 * enqueued there, and waits for the stream.  This is the one call of the
 * library that synchronizes.  *status gets BSQ_DEV_OK or the first
 * BSQ_DEV_* value a kernel recorded; the word itself is left as it is, so
 * the caller zeroes it before reusing it.  Returns BSQ_ERR_NULL if either
 * pointer is NULL and BSQ_ERR_CUDA if the copy or the wait fails (an earlier
 * asynchronous CUDA error of the stream included). */
bsq_status bsq_check_status(const int32_t* dev_status, int32_t* status, bsq_stream_t stream);

/* ---------------------------------------------------------------------------
 * quantize_nvfp4_per_token: per-row (per-token) NVFP4 quantization.
 * "4ビットの教訓" (hackernews.jp), "ベースラインレシピ": each token computes its
 * own FP32 activation scale over the hidden dimension, online, and the
 * quantization kernel emits packed FP4 values, E4M3 block scales and the FP32
 * token scales in one pass; "LMSYS Drops Miles ...", "Recipe 2: Per-token
 * NVFP4 for MoE experts".  "4/6" ("End-to-End 4-Bit Training", "工程细节"):
 * per block, the lower-error of two candidate scales.
 *   x          bf16 [rows][ldx], K columns used; ldx % 8 == 0
 *   codes      out, [rows][K/2]
 *   sf         out, E4M3 block scales, linear [rows][K/16] or swizzled
 *   row_scale  out, fp32 [rows]: t = amax(|x_row|) / 2688 (6 * 448)
 *   flags      BSQ_SF_SWIZZLED, BSQ_FOUR_SIX
 * K % 16 == 0, 0 < K <= 65536; rows >= 0 (0 is a no-op).
 * ------------------------------------------------------------------------- */
bsq_status quantize_nvfp4_per_token(const void* x, int64_t rows, int64_t K, int64_t ldx,
                                    uint8_t* codes, uint8_t* sf, float* row_scale,
                                    uint32_t flags, int32_t* dev_status, bsq_stream_t stream);

/* ---------------------------------------------------------------------------
 * quantize_nvfp4_per_expert: NVFP4 weights with one FP32 scale per expert
 * ("4ビットの教訓", "ベースラインレシピ": weights use the standard format with
 * one global FP32 scale; "End-to-End 4-Bit Training", "工程细节": per-expert
 * outer scale).  For SwiGLU gate/up weights pass the concatenated [2I][H]
 * matrix per expert so gate and up share one scale ("Miles Blackwell RL ...",
 * "Un quantizzatore condiviso è il vero meccanismo").  No 4/6 on weights.
 *   w             bf16 [experts][rows][K], contiguous
 *   codes         out, [experts][rows][K/2]
 *   sf            out, linear [experts*rows][K/16] or swizzled over the
 *                 experts*rows stacked rows (rows % 128 == 0 when swizzled)
 *   expert_scale  out, fp32 [experts]; also used as scratch during the call
 * ------------------------------------------------------------------------- */
bsq_status quantize_nvfp4_per_expert(const void* w, int64_t experts, int64_t rows, int64_t K,
                                     uint8_t* codes, uint8_t* sf, float* expert_scale,
                                     uint32_t flags, int32_t* dev_status, bsq_stream_t stream);

/* ---------------------------------------------------------------------------
 * quantize_nvfp4_rht: per-token NVFP4 of a 32-point random Hadamard transform
 * of each row ("End-to-End 4-Bit Training", "第三个决定": a 32-dimensional
 * random Hadamard transform spreads outliers over their group before block
 * quantization; the page quantizes the result to a format it does not
 * define, NVFP4 stands in).  Per group of 32 consecutive elements,
 * y = H32 (s . x): H32 the Sylvester Hadamard matrix (entries +-1,
 * H[i][j] = (-1)^popcount(i & j)), unnormalized (H32 H32 = 32 I inverts it),
 * computed in binary32 by the butterfly h = 1, 2, 4, 8, 16 ((v_i, v_{i+h}) <-
 * (v_i + v_{i+h}, v_i - v_{i+h}) for (i & h) == 0); s_j = -1 iff bit j of
 * word 0 of Philox4x32-10(key = seed, counter = (0, 0, 2, 0)).  Then the
 * per-token recipe of quantize_nvfp4_per_token on y (no 4/6).
 *   x          bf16 [rows][ldx], K columns used; ldx % 8 == 0, 16-byte aligned
 *   codes      out, [rows][K/2] (codes of y)
 *   sf         out, E4M3 block scales of y, linear or swizzled
 *   row_scale  out, fp32 [rows]
 *   flags      BSQ_SF_SWIZZLED
 * K % 32 == 0, 0 < K <= 65536; rows >= 0 (0 is a no-op).
 * ------------------------------------------------------------------------- */
bsq_status quantize_nvfp4_rht(const void* x, int64_t rows, int64_t K, int64_t ldx, uint64_t seed,
                              uint8_t* codes, uint8_t* sf, float* row_scale,
                              uint32_t flags, int32_t* dev_status, bsq_stream_t stream);

/* ---------------------------------------------------------------------------
 * quantize_nvfp4_2d: NVFP4 with one E4M3 scale per 16 x 16 square block and
 * one FP32 scale per tensor, emitting the row-major operand and, optionally,
 * the transposed one ("End-to-End 4-Bit Training", "第二个决定": square block
 * scales are the same before and after the transpose, so the backward
 * operand needs no requantization; the page's authors found 256 values per
 * scale too coarse next to outliers and requantized instead).
 * t = amax(|x|) / 2688 over the whole tensor; per tile, the per-row recipe's
 * block steps with the tile's maximum: s = E4M3(amax_tile / (6 t)),
 * d = s * t, code = E2M1(x * (1 / d)).  t == 0 gives all-zero codes and scales.
 *   x            bf16 [rows][K], contiguous, 16-byte aligned
 *   codes        out, [rows][K/2] (low nibble = even column), 16-byte aligned
 *   sf_tiles     out, E4M3 [rows/16][K/16] (linear)
 *   codes_t      out, [K][rows/2]: the codes of x^T, 8-byte aligned (NULL:
 *                skip, with sf_tiles_t)
 *   sf_tiles_t   out, E4M3 [K/16][rows/16] (= sf_tiles transposed)
 *   tensor_scale out, fp32 [1]
 * rows % 16 == 0, K % 16 == 0, 0 < K <= 65536; rows == 0 is a no-op.
 * flags must be 0.  The result equals quantizing x^T with the same recipe.
 * ------------------------------------------------------------------------- */
bsq_status quantize_nvfp4_2d(const void* x, int64_t rows, int64_t K,
                             uint8_t* codes, uint8_t* sf_tiles,
                             uint8_t* codes_t, uint8_t* sf_tiles_t, float* tensor_scale,
                             uint32_t flags, int32_t* dev_status, bsq_stream_t stream);

/* ---------------------------------------------------------------------------
 * dequantize_nvfp4: BF16 reconstruction of NVFP4 operands, for the
 * dequantized backward mode ("LMSYS Drops Miles ...", "Recipe 2: Per-token
 * NVFP4 for MoE experts"; "Miles Blackwell RL ...", "Un quantizzatore
 * condiviso ...": the backward GEMMs run in BF16 on BF16 operands rebuilt
 * from the exact low-precision values of the forward pass).  Per element
 * y = bf16_rn(rn(rn(e2m1(code) * e4m3(sf)) * t)) in binary32, t the FP32
 * scale of the element's row (activations, group_rows = 1) or of its group of
 * group_rows consecutive rows (per-expert weights, group_rows = rows of one
 * expert).  The inner product is exact; bf16_rn is round-to-nearest-even.
 *   codes  [rows][K/2] (low nibble = even element), 16-byte aligned
 *   sf     E4M3 block scales, linear [rows][K/16] or swizzled (BSQ_SF_SWIZZLED;
 *          the buffer covers rows padded to 128), 4-byte aligned
 *   scale  fp32 [rows] (group_rows = 1) or [ceil(rows / group_rows)]
 *   y      out, bf16 [rows][ldy], K columns written; ldy >= K, ldy % 8 == 0,
 *          16-byte aligned
 * K % 16 == 0, 0 < K <= 65536; rows >= 0 (0 is a no-op).  E4M3 NaN codes
 * are outside the contract.  All pointers are device pointers owned by the
 * caller; the call only enqueues on `stream`.
 * ------------------------------------------------------------------------- */
bsq_status dequantize_nvfp4(const uint8_t* codes, const uint8_t* sf, const float* scale,
                            int64_t rows, int64_t K, int64_t group_rows,
                            void* y, int64_t ldy, uint32_t flags, int32_t* dev_status,
                            bsq_stream_t stream);

/* ---------------------------------------------------------------------------
 * quantize_mxfp8_rowcol: MXFP8 row-wise and column-wise copies of one bf16
 * tensor in one pass, both from the original values ("LMSYS Drops Miles ...",
 * "Recipe 1: End-to-end MXFP8"; "Miles Blackwell RL ...", "Un quantizzatore
 * condiviso ...": blocks follow the reduction dimension).  Shared exponent:
 * X = clamp(floor(log2(amax)) - 8, -127, 127), SF = X + 127, codes =
 * E4M3(x * 2^-X), round to nearest even, saturating at 448.
 *   x          bf16 [rows][ldx]; rows % 32 == 0, K % 32 == 0, ldx % 8 == 0;
 *              x and the code buffers 16-byte aligned, the SF buffers 4-byte
 *              aligned (else BSQ_ERR_ALIGN)
 *   row_codes  out, E4M3 [rows][K] (NULL: skip the row copy with row_sf)
 *   row_sf     out, E8M0 [rows][K/32] linear or swizzled
 *   col_codes  out, E4M3 [K][rows] (the column copy, stored transposed;
 *              NULL: skip with col_sf)
 *   col_sf     out, E8M0 [K][rows/32] linear or swizzled
 *   flags      BSQ_SF_SWIZZLED
 * ------------------------------------------------------------------------- */
bsq_status quantize_mxfp8_rowcol(const void* x, int64_t rows, int64_t K, int64_t ldx,
                                 uint8_t* row_codes, uint8_t* row_sf,
                                 uint8_t* col_codes, uint8_t* col_sf,
                                 uint32_t flags, int32_t* dev_status, bsq_stream_t stream);

/* ---------------------------------------------------------------------------
 * requant_transpose_sr: backward requantization ("End-to-End 4-Bit Training",
 * "第二个决定": dequantize the forward tensor, transpose, quantize again with
 * stochastic rounding).  D = dequant(input) in binary32; Y = D^T [K][rows];
 * targets:
 *   NVFP4: each row of Y with the per-row recipe of quantize_nvfp4_per_token
 *          (its own FP32 scale over the whole row; no 4/6);
 *   MXFP8: each row of Y with the rule of quantize_mxfp8_rowcol.
 * BSQ_STOCHASTIC rounds element codes stochastically with 16 random bits per
 * element: Philox4x32-10, key = seed, counter = (idx/8, stream, 0) with idx
 * the element's linear index in Y and stream 0 (NVFP4) / 1 (MXFP8); element
 * idx uses the 16-bit half idx%2 of word (idx/2)%4; round up iff
 * bits < 65536 * (|v| - lo) / (hi - lo).  Scales are always round-to-nearest.
 *   codes, sf, row_scale   the NVFP4 input [rows][K] (sf per `flags`)
 *   nv_*                   out NVFP4 of Y: codes [K][rows/2], sf, scale [K]
 *                          (all three NULL: skip this target)
 *   mx_*                   out MXFP8 of Y: codes [K][rows], sf [K][rows/32]
 *                          (both NULL: skip)
 *   workspace              device scratch of bsq_requant_workspace_size()
 *                          bytes (the column maxima of |D|); may be NULL
 *                          when that size is 0
 * rows % 32 == 0, K % 16 == 0; codes and the output codes 16-byte aligned,
 * the SF buffers (input and outputs) 4-byte aligned (else BSQ_ERR_ALIGN).
 * ------------------------------------------------------------------------- */
size_t bsq_requant_workspace_size(int64_t rows, int64_t K, int32_t nvfp4_target);
bsq_status requant_transpose_sr(const uint8_t* codes, const uint8_t* sf, const float* row_scale,
                                int64_t rows, int64_t K,
                                uint8_t* nv_codes_T, uint8_t* nv_sf_T, float* nv_scale_T,
                                uint8_t* mx_codes_T, uint8_t* mx_sf_T,
                                uint64_t seed, void* workspace, size_t workspace_bytes,
                                uint32_t flags, int32_t* dev_status, bsq_stream_t stream);

/* ---------------------------------------------------------------------------
 * requant_transpose_sr_noalloc: requant_transpose_sr for callers that cannot
 * hand the library device scratch memory -- a host framework that owns only
 * its input and output buffers, or code that must not allocate device memory
 * once it is running.  (The source pages have no counterpart; this is an
 * interface convenience.)  Same arguments, layouts and results as
 * requant_transpose_sr, without the workspace: the column maxima of the
 * NVFP4 target live in a 256 KB array inside the library that every GPU
 * loading the library keeps until the process exits.  The function calls no
 * allocator.
 *   - K must be <= 65536; larger K is rejected with BSQ_ERR_SHAPE before
 *     anything is enqueued.
 *   - The first call on each device looks up the array's device address
 *     (with that device current); make that first call before capturing the
 *     stream into a graph.  The address is kept for the life of the process,
 *     so the function is not supported after cudaDeviceReset (which unloads
 *     the library's device code) in the same process.
 *   - Every call on a device uses the same array and clears the part it
 *     needs first; calls whose GPU work overlaps (other streams, other host
 *     threads on the same device) race on it and must be serialized by the
 *     caller.
 * ------------------------------------------------------------------------- */
bsq_status requant_transpose_sr_noalloc(const uint8_t* codes, const uint8_t* sf, const float* row_scale,
                                        int64_t rows, int64_t K,
                                        uint8_t* nv_codes_T, uint8_t* nv_sf_T, float* nv_scale_T,
                                        uint8_t* mx_codes_T, uint8_t* mx_sf_T,
                                        uint64_t seed, uint32_t flags, int32_t* dev_status, bsq_stream_t stream);

/* ---------------------------------------------------------------------------
 * grouped_expert_gemm_fp4: block-scaled grouped GEMM on the tensor cores
 * (kind::mxf4nvf4, E4M3 scale per 16 elements) with the FP32 rescale fused in
 * the epilogue ("LMSYS Drops Miles ...", "Why Blackwell changes the math":
 * rescaling in hardware; "Results": per-token FP32 scaling belongs in the GEMM
 * epilogue).  For each expert e the rows [offsets[e], offsets[e+1]) of A are
 * multiplied by expert e's B:
 *   y[m][n] = sum_k A[m][k] * B[e][n][k] * a_scale[m] * b_scale[e]
 *   a_codes, a_sf   A, NVFP4 [m_capacity][K/2], SF swizzled (rows padded to
 *                   128) -- per-token scales a_scale [m_capacity]
 *   offsets         device int32 [experts+1], ascending; every segment
 *                   start offsets[e] (e < experts) is a multiple of 128, the
 *                   total offsets[experts] may be any value <= m_capacity
 *   b_codes, b_sf   B, NVFP4 [experts][N][K/2], SF swizzled over the
 *                   experts*N stacked rows -- b_scale [experts]
 *   epilogue        BSQ_EPI_F32 / BSQ_EPI_BF16 (out [m_capacity][ldo]) or
 *                   BSQ_EPI_SWIGLU_BF16 (out [m_capacity][ldo], N/2 columns
 *                   used: B rows [0,N/2) are gate, [N/2,N) are up)
 * K % 64 == 0; N % 128 == 0 (N % 256 == 0 for SwiGLU).  Rows of a segment
 * past the routed rows are computed like any other row.
 * ------------------------------------------------------------------------- */
bsq_status grouped_expert_gemm_fp4(const uint8_t* a_codes, const uint8_t* a_sf,
                                   const float* a_scale, const int32_t* offsets,
                                   int64_t experts, int64_t m_capacity, int64_t K, int64_t N,
                                   const uint8_t* b_codes, const uint8_t* b_sf,
                                   const float* b_scale, int32_t epilogue,
                                   void* out, int64_t ldo,
                                   uint32_t flags, int32_t* dev_status, bsq_stream_t stream);

/* ---------------------------------------------------------------------------
 * grouped_expert_gemm_mxfp8: the same grouped GEMM on MXFP8 operands
 * (kind::mxf8f6f4 with one E8M0 scale per 32 elements), for the backward
 * GEMMs of the MXFP8 recipe ("Miles Blackwell RL ...", "Il supporto Miles
 * ...": the weight- and data-gradient GEMMs run in MXFP8 too; "LMSYS Drops
 * Miles ...", "Recipe 1: End-to-end MXFP8"), fed by the row copies of
 * quantize_mxfp8_rowcol and the MXFP8 targets of requant_transpose_sr:
 *   y[m][n] = sum_k A[m][k] * B[e][n][k] * a_scale[m] * b_scale[e]
 * with A[m][k] = E4M3(code) * 2^(E8M0(sf) - 127) (and B likewise); pass ones
 * as a_scale / b_scale for plain MXFP8.
 *   a_codes, a_sf   A, E4M3 [m_capacity][K], E8M0 SF swizzled (rows padded
 *                   to 128)
 *   offsets         as for grouped_expert_gemm_fp4
 *   b_codes, b_sf   B, E4M3 [experts][N][K], SF swizzled over the experts*N
 *                   stacked rows
 *   epilogue        BSQ_EPI_F32 or BSQ_EPI_BF16 (out [m_capacity][ldo])
 * K % 128 == 0; N % 128 == 0.
 * ------------------------------------------------------------------------- */
bsq_status grouped_expert_gemm_mxfp8(const uint8_t* a_codes, const uint8_t* a_sf,
                                     const float* a_scale, const int32_t* offsets,
                                     int64_t experts, int64_t m_capacity, int64_t K, int64_t N,
                                     const uint8_t* b_codes, const uint8_t* b_sf,
                                     const float* b_scale, int32_t epilogue,
                                     void* out, int64_t ldo,
                                     uint32_t flags, int32_t* dev_status, bsq_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_expert_forward: routed-expert SwiGLU MLP with NVFP4 activations and
 * weights, one GPU:
 *   1. route: count rows per expert, pad each expert's segment to 128 rows,
 *      slots in ascending (token, k) order;
 *   2. per-token NVFP4 quantization of x into the routed slots;
 *   3. grouped GEMM with gate/up weights and the fused SwiGLU + FP32 rescale
 *      epilogue -> h (bf16);
 *   4. per-token NVFP4 quantization of h (4/6 with BSQ_FOUR_SIX).  With
 *      BSQ_MOE_FUSED_H, step 3's epilogue does it instead: once all of a
 *      row's N tiles are done on the CTA it quantizes the row from the
 *      CTA's scratch, so h never reaches memory ("LMSYS Drops Miles ...",
 *      section "Results": the per-token scaling inside the GEMM).  Same
 *      results bit for bit; on GB300 it measured slower (the quantization
 *      then runs on the 16 epilogue warps, already GEMM1's bottleneck,
 *      instead of the whole GPU);
 *   5. grouped GEMM with down weights, rescale -> per-slot outputs (bf16);
 *   6. combine: y[t] = sum_j w[t][j] * out[slot(t, j)], fp32, j ascending.
 *   x              bf16 [T][H]
 *   topk_ids       int32 [T][topk], values in [0, E)
 *   topk_weights   fp32 [T][topk]
 *   wgu_*          gate/up weights NVFP4 [E][2I][H/2], SF swizzled, scale [E]
 *   wd_*           down weights NVFP4 [E][H][I/2], SF swizzled, scale [E]
 *   y              out bf16 [T][H]
 *   workspace      device scratch, bsq_moe_workspace_size() bytes; its
 *                  sub-buffers (bsq_moe_layout) hold the intermediates
 *   flags          BSQ_FOUR_SIX (the 4/6 choice on x and h); BSQ_MOE_FUSED_H
 *                  (above), and with it BSQ_MOE_KEEP_H, which also keeps the
 *                  whole bf16 h in the layout's h buffer (for checking the
 *                  stages separately), otherwise untouched in that mode
 * H % 256 == 0, I % 128 == 0, topk <= 32; BSQ_MOE_FUSED_H on a device with
 * more than BSQ_MOE_MAX_CTAS SMs is refused (BSQ_ERR_UNSUPPORTED).
 * ------------------------------------------------------------------------- */
#define BSQ_MOE_MAX_CTAS 256  /* GEMM1 CTAs the h scratch is sized for */
typedef struct {
    size_t offsets;      /* int32 [E+1]   padded segment starts */
    size_t counts;       /* int32 [E]     routed rows per expert */
    size_t slot_of;      /* int32 [T*topk] row of routed pair (t, j) */
    size_t row_src;      /* int32 [cap]   t*topk + j, or -1 for padding */
    size_t xq_codes;     /* u8 [cap][H/2] */
    size_t xq_sf;        /* u8 swizzled, cap x H/16 */
    size_t xq_scale;     /* fp32 [cap] */
    size_t h;            /* bf16 [cap][I] (with BSQ_MOE_FUSED_H, only with BSQ_MOE_KEEP_H) */
    size_t hq_codes;     /* u8 [cap][I/2] */
    size_t hq_sf;        /* u8 swizzled, cap x I/16 */
    size_t hq_scale;     /* fp32 [cap] */
    size_t out;          /* bf16 [cap][H] per-slot expert outputs */
    size_t scan;         /* int32 scratch for the routing scan: per-512-pair
                            chunk expert histograms and a counter */
    size_t h_scratch;    /* bf16 [BSQ_MOE_MAX_CTAS][2][128][I]: with
                            BSQ_MOE_FUSED_H, each GEMM1 CTA's rows of h (two
                            units) between the SwiGLU and their quantization
                            (stays in L2) */
    size_t total;        /* bytes */
    int64_t capacity;    /* cap: T*topk + E*127 rounded up to 128 */
} bsq_moe_layout;

size_t bsq_moe_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk);
bsq_status bsq_moe_workspace_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk,
                                    bsq_moe_layout* layout);
bsq_status moe_expert_forward(const void* x, int64_t T, int64_t H, int64_t I, int64_t E, int64_t topk,
                              const int32_t* topk_ids, const float* topk_weights,
                              const uint8_t* wgu_codes, const uint8_t* wgu_sf, const float* wgu_scale,
                              const uint8_t* wd_codes, const uint8_t* wd_sf, const float* wd_scale,
                              void* y, void* workspace, size_t workspace_bytes,
                              uint32_t flags, int32_t* dev_status, bsq_stream_t stream);

/* ---------------------------------------------------------------------------
 * bsq_set_stage_events: profiling hook for moe_expert_forward.  While set
 * (events != NULL, n >= 7), every moe_expert_forward call made from the
 * calling host thread records events[0..6] (cudaEvent_t handles owned by the
 * caller) on its stream: before routing, after routing, after the
 * quantize-scatter, after GEMM1, after the quantization of h, after GEMM2,
 * after the combine.  The array must stay valid while set; pass NULL to
 * clear.  Returns BSQ_ERR_SHAPE if 0 < n < 7.
 * ------------------------------------------------------------------------- */
bsq_status bsq_set_stage_events(void* const* events, int32_t n);

/* ---------------------------------------------------------------------------
 * Helpers (also used by the tests).
 * bsq_sf_swizzle / bsq_sf_unswizzle: convert an SF matrix [rows][cols]
 * between the linear and the swizzled layout (swizzled padding set to 0).
 * bsq_format_probe: element-format conversions exactly as the kernels do
 * them: kind 0 = E2M1 RNE, 1 = E4M3 RNE satfinite, 2 = E2M1 stochastic,
 * 3 = E4M3 stochastic (rbits[i] & 0xFFFF are the random bits), 4 = E2M1
 * decode (in: code in the low byte of the float's bits), 5 = E4M3 decode.
 * Output: one byte (kinds 0-3) or one float (kinds 4-5) per element.
 * bsq_philox_bits16: the 16 random bits element idx0+i receives from
 * (seed, stream), for i < n, as uint16 values.
 * ------------------------------------------------------------------------- */
bsq_status bsq_sf_swizzle(const uint8_t* sf_linear, int64_t rows, int64_t cols,
                          uint8_t* sf_swizzled, bsq_stream_t stream);
bsq_status bsq_sf_unswizzle(const uint8_t* sf_swizzled, int64_t rows, int64_t cols,
                            uint8_t* sf_linear, bsq_stream_t stream);
bsq_status bsq_format_probe(int32_t kind, const float* in, const uint32_t* rbits,
                            void* out, int64_t n, bsq_stream_t stream);
bsq_status bsq_philox_bits16(uint64_t seed, uint32_t stream_id, uint64_t idx0, int64_t n,
                             uint16_t* out, bsq_stream_t stream);

/* ---------------------------------------------------------------------------
 * bsq_mma_ceiling: measures the tensor cores' block-scaled MMA ceiling, the
 * denominator of the grouped GEMM's roofline fraction (the pages give only
 * nominal FP4 throughputs: "End-to-End 4-Bit Training", section "先说为什么难").
 * One CTA per SM issues `iters` back-to-back MMAs of the GEMM's own form from
 * operands already in shared memory, scale factors already in tensor memory:
 *   fmt        0 = NVFP4 (kind::mxf4nvf4 scale_vec::4X, 128 x 256 x 64 per CTA),
 *              1 = MXFP8 (kind::mxf8f6f4 scale_vec::1X, 128 x 256 x 32 per CTA)
 *   cta_group  1 = one CTA per MMA; 2 = clusters of two CTAs sharing one
 *              256 x 256 MMA (cta_group::2)
 *   iters      MMAs per CTA, 1..65536
 *   cycles     device uint64 [number of SMs]: for each issuing CTA the
 *              clock64 cycles from its first issue to the completion of its
 *              last MMA; 0 for the second CTA of a pair
 *   ctas       host out: the number of CTAs launched (the SMs, rounded down
 *              to a multiple of cta_group)
 * The caller times the launch (CUDA events) for the FLOP rate:
 * ctas * iters * 2 * 128 * 256 * K FLOPs.  A wait that runs out is reported
 * in dev_status as BSQ_DEV_TIMEOUT.
 * ------------------------------------------------------------------------- */
bsq_status bsq_mma_ceiling(int32_t fmt, int32_t cta_group, int32_t iters, uint64_t* cycles, int32_t* ctas,
                           int32_t* dev_status, bsq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* BSQ_H */
