"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function include/bsq.h declares, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "bsq.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+\**([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "return")))


@pytest.fixture(scope="module")
def lib():
    import block_scaled_precision_quantize_gb300 as bsq
    bsq.build()
    return bsq.load()


def test_header_declares_the_five_hot_path_entry_points():
    names = declared_functions()
    for n in ("quantize_nvfp4_per_token", "quantize_mxfp8_rowcol", "requant_transpose_sr",
              "grouped_expert_gemm_fp4", "moe_expert_forward"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_validation_without_a_gpu(lib):
    import block_scaled_precision_quantize_gb300 as bsq
    P = ctypes.c_void_p
    dummy = P(4096)
    word = ctypes.c_int32(-1)
    assert lib.bsq_check_status(None, ctypes.byref(word), None) == 1  # null status word
    assert lib.bsq_check_status(dummy, None, None) == 1               # null destination
    assert word.value == -1                                            # nothing written
    st = lib.quantize_nvfp4_per_token(dummy, 8, 256, 256, dummy, dummy, dummy, 1 << 7, None, None)
    assert st == 4  # flags
    st = lib.quantize_nvfp4_per_token(dummy, 8, 250, 256, dummy, dummy, dummy, 0, None, None)
    assert st == 2  # K % 16
    st = lib.quantize_nvfp4_per_token(None, 8, 256, 256, dummy, dummy, dummy, 0, None, None)
    assert st == 1  # null
    st = lib.quantize_nvfp4_per_token(P(4100), 8, 256, 256, dummy, dummy, dummy, 0, None, None)
    assert st == 3  # alignment
    st = lib.quantize_nvfp4_per_token(dummy, 0, 256, 256, dummy, dummy, dummy, 0, None, None)
    assert st == 0  # empty input is a no-op
    st = lib.quantize_mxfp8_rowcol(dummy, 48, 256, 256, dummy, dummy, dummy, dummy, 0, None, None)
    assert st == 2  # rows % 32
    st = lib.requant_transpose_sr(dummy, dummy, dummy, 64, 256, dummy, dummy, dummy, None, None, 0, None, 0,
                                  bsq.STOCHASTIC, None, None)
    assert st == 7  # workspace required for the NVFP4 target
    st = lib.grouped_expert_gemm_fp4(dummy, dummy, dummy, dummy, 2, 256, 96, 256, dummy, dummy, dummy, 0,
                                     dummy, 256, bsq.SF_SWIZZLED, None, None)
    assert st == 2  # K % 64
    st = lib.grouped_expert_gemm_fp4(dummy, dummy, dummy, dummy, 2, 256, 256, 384, dummy, dummy, dummy,
                                     bsq.EPI_SWIGLU_BF16, dummy, 192, bsq.SF_SWIZZLED, None, None)
    assert st == 2  # SwiGLU needs N % 256
    st = lib.moe_expert_forward(dummy, 16, 2048, 768, 8, 40, dummy, dummy, dummy, dummy, dummy, dummy, dummy,
                                dummy, dummy, dummy, 1 << 30, 0, None, None)
    assert st == 2  # topk > 32
    st = lib.moe_expert_forward(dummy, 16, 2048, 768, 8, 4, dummy, dummy, dummy, dummy, dummy, dummy, dummy,
                                dummy, dummy, dummy, 16, 0, None, None)
    assert st == 7  # workspace too small


def test_moe_workspace_layout_is_consistent(lib):
    import block_scaled_precision_quantize_gb300 as bsq
    T, H, I, E, k = 16384, 2048, 768, 128, 8
    L = bsq.moe_workspace_layout(T, H, I, E, k)
    assert L.capacity % 128 == 0 and L.capacity >= T * k + E * 127
    fields = ["offsets", "counts", "slot_of", "row_src", "xq_codes", "xq_sf", "xq_scale", "h", "hq_codes",
              "hq_sf", "hq_scale", "out", "scan"]
    offs = [getattr(L, f) for f in fields]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert L.h - L.xq_codes >= L.capacity * (H // 2 + H // 16 + 4)
    assert L.total == bsq.moe_workspace_size(T, H, I, E, k) and L.total > L.scan


def test_host_validation_of_dequantize_and_2d_without_a_gpu(lib):
    P = ctypes.c_void_p
    d = P(4096)
    # dequantize_nvfp4(codes, sf, scale, rows, K, group_rows, y, ldy, flags, status, stream)
    assert lib.dequantize_nvfp4(d, d, d, 8, 256, 1, d, 256, 1 << 5, None, None) == 4  # flags
    assert lib.dequantize_nvfp4(d, d, d, 8, 250, 1, d, 256, 0, None, None) == 2       # K % 16
    assert lib.dequantize_nvfp4(d, d, d, 8, 256, 1, d, 128, 0, None, None) == 2       # ldy < K
    assert lib.dequantize_nvfp4(d, d, d, 8, 256, 0, d, 256, 0, None, None) == 2       # group_rows
    assert lib.dequantize_nvfp4(None, d, d, 8, 256, 1, d, 256, 0, None, None) == 1    # null
    assert lib.dequantize_nvfp4(d, d, d, 8, 256, 1, P(4104), 256, 0, None, None) == 3  # y alignment
    assert lib.dequantize_nvfp4(d, d, d, 8, 256, 1, d, 260, 0, None, None) == 3       # ldy % 8
    assert lib.dequantize_nvfp4(d, P(4097), d, 8, 256, 1, d, 256, 0, None, None) == 3  # sf alignment
    assert lib.dequantize_nvfp4(d, d, d, 0, 256, 1, d, 256, 0, None, None) == 0       # empty: no-op
    # quantize_nvfp4_2d(x, rows, K, codes, sf, codes_t, sf_t, scale, flags, status, stream)
    assert lib.quantize_nvfp4_2d(d, 32, 256, d, d, d, d, d, 1, None, None) == 4        # flags
    assert lib.quantize_nvfp4_2d(d, 24, 256, d, d, d, d, d, 0, None, None) == 2        # rows % 16
    assert lib.quantize_nvfp4_2d(d, 32, 248, d, d, d, d, d, 0, None, None) == 2        # K % 16
    assert lib.quantize_nvfp4_2d(d, 32, 256, d, d, d, None, d, 0, None, None) == 1     # transposed pair half given
    assert lib.quantize_nvfp4_2d(d, 32, 256, d, d, None, None, None, 0, None, None) == 1  # no scale
    assert lib.quantize_nvfp4_2d(P(4100), 32, 256, d, d, d, d, d, 0, None, None) == 3  # x alignment
    assert lib.quantize_nvfp4_2d(d, 32, 256, d, d, P(4100), d, d, 0, None, None) == 3  # codes_t alignment
    assert lib.quantize_nvfp4_2d(d, 0, 256, d, d, d, d, d, 0, None, None) == 0         # empty: no-op


def test_host_validation_of_rht_and_mxfp8_gemm_without_a_gpu(lib):
    P = ctypes.c_void_p
    d = P(4096)
    # quantize_nvfp4_rht(x, rows, K, ldx, seed, codes, sf, scale, flags, status, stream)
    assert lib.quantize_nvfp4_rht(d, 8, 256, 256, 7, d, d, d, 1 << 6, None, None) == 4  # flags
    assert lib.quantize_nvfp4_rht(d, 8, 48, 48, 7, d, d, d, 0, None, None) == 2         # K % 32
    assert lib.quantize_nvfp4_rht(d, 8, 256, 128, 7, d, d, d, 0, None, None) == 2       # ldx < K
    assert lib.quantize_nvfp4_rht(None, 8, 256, 256, 7, d, d, d, 0, None, None) == 1    # null
    assert lib.quantize_nvfp4_rht(P(4100), 8, 256, 256, 7, d, d, d, 0, None, None) == 3  # alignment
    assert lib.quantize_nvfp4_rht(d, 0, 256, 256, 7, d, d, d, 0, None, None) == 0       # empty: no-op
    # grouped_expert_gemm_mxfp8(a, asf, ascale, offsets, E, M, K, N, b, bsf, bscale, epi, out, ldo, flags, st, s)
    assert lib.grouped_expert_gemm_mxfp8(d, d, d, d, 1, 128, 192, 128, d, d, d, 0, d, 128, 1, None, None) == 2  # K % 128
    assert lib.grouped_expert_gemm_mxfp8(d, d, d, d, 1, 128, 256, 96, d, d, d, 0, d, 128, 1, None, None) == 2   # N % 128
    assert lib.grouped_expert_gemm_mxfp8(d, d, d, d, 1, 128, 256, 128, d, d, d, 2, d, 128, 1, None, None) == 4  # no SwiGLU
    assert lib.grouped_expert_gemm_mxfp8(d, d, d, d, 1, 128, 256, 128, d, d, d, 0, d, 64, 1, None, None) == 2   # ldo < N
    assert lib.grouped_expert_gemm_mxfp8(d, d, None, d, 1, 128, 256, 128, d, d, d, 0, d, 128, 1, None, None) == 1
    assert lib.grouped_expert_gemm_mxfp8(d, d, d, d, 1, 0, 256, 128, d, d, d, 0, d, 128, 1, None, None) == 0     # empty
