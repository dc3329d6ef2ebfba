"""The oracle: a plain single-threaded CPU implementation of the block-scaled
quantization hot path (``bsq_oracle.c``), loaded through ctypes.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product library
never does. It shares no code with the CUDA path; both sides only share the
seeded input generators, which hold none of the method's arithmetic.

Every function takes and returns numpy arrays. bf16 tensors are passed as
their raw uint16 bit patterns. Scale factors come back in the linear layout
[rows][K/16] (NVFP4) or [rows][K/32] (MXFP8).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsq_oracle.c")
_HDR = os.path.join(_HERE, "bsq_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libbsq_oracle.so")
# IEEE binary32 semantics: one rounding per operation, no contraction into
# FMA, no fast math, no flush-to-zero.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fvisibility=hidden", "-Wall", "-Wextra", "-Wno-unused-parameter"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build (idempotent)."""
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64
_U32 = ctypes.c_uint32
_INT = ctypes.c_int


def _declare(L):
    sig = {
        "bsqo_e2m1_decode": (ctypes.c_float, [_U32]),
        "bsqo_e2m1_encode": (_U32, [ctypes.c_float]),
        "bsqo_e2m1_encode_sr": (_U32, [ctypes.c_float, _U32]),
        "bsqo_e4m3_decode": (ctypes.c_float, [_U32]),
        "bsqo_e4m3_encode": (_U32, [ctypes.c_float]),
        "bsqo_e4m3_encode_sr": (_U32, [ctypes.c_float, _U32]),
        "bsqo_e8m0_decode": (ctypes.c_float, [_U32]),
        "bsqo_e2m1_encode_array": (None, [_P, _I64, _P]),
        "bsqo_e4m3_encode_array": (None, [_P, _I64, _P]),
        "bsqo_philox4x32_10": (None, [_P, _P, _P]),
        "bsqo_sr_bits16": (_U32, [_U64, _U32, _U64]),
        "bsqo_nvfp4_quantize_rows": (None, [_P, _I64, _I64, _I64, _INT, _P, _P, _P]),
        "bsqo_nvfp4_quantize_rows_given_t": (None, [_P, _I64, _I64, _P, _INT, _P, _P]),
        "bsqo_nvfp4_quantize_group": (None, [_P, _I64, _I64, _I64, _P, _P, _P]),
        "bsqo_nvfp4_dequantize": (None, [_P, _P, _P, _I64, _I64, _P]),
        "bsqo_nvfp4_quantize_2d": (None, [_P, _I64, _I64, _P, _P, _P]),
        "bsqo_rht_signs": (_U32, [_U64]),
        "bsqo_rht32": (None, [_P, _I64, _U32, _P]),
        "bsqo_nvfp4_quantize_rht": (None, [_P, _I64, _I64, _U64, _P, _P, _P]),
        "bsqo_nvfp4_block_candidate": (None, [_P, ctypes.c_float, ctypes.c_float, _P, _P, _P]),
        "bsqo_sf_swizzled_offset": (_I64, [_I64, _I64, _I64]),
        "bsqo_sf_swizzle": (None, [_P, _I64, _I64, _P]),
        "bsqo_mxfp8_quantize_rowcol": (None, [_P, _I64, _I64, _I64, _P, _P, _P, _P]),
        "bsqo_requant_transpose": (None, [_P, _P, _P, _I64, _I64, _INT, _U64, _P, _P, _P, _P, _P]),
        "bsqo_gemm_nvfp4": (None, [_P, _P, _P, _I64, _I64, _P, _P, ctypes.c_float, _I64, _P, _P]),
        "bsqo_gemm_mxfp8": (None, [_P, _P, _P, _I64, _I64, _P, _P, ctypes.c_float, _I64, _P, _P]),
        "bsqo_gemm_nvfp4_sampled": (None, [_P, _P, _P, _I64, _P, _P, _P, _P, _P, _P, _I64, _P, _P]),
        "bsqo_route": (_I64, [_P, _I64, _I64, _I64, _I64, _P, _P, _P]),
        "bsqo_swiglu": (None, [_P, _I64, _I64, _P]),
        "bsqo_combine": (None, [_P, _I64, _P, _P, _I64, _I64, _P]),
        "bsqo_f64_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
        "bsqo_f64_to_bf16_array": (None, [_P, _I64, _P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- formats
def e2m1_decode(code: int) -> float:
    return lib().bsqo_e2m1_decode(int(code))


def e2m1_encode(v: float) -> int:
    return lib().bsqo_e2m1_encode(float(v))


def e2m1_encode_sr(v: float, r16: int) -> int:
    return lib().bsqo_e2m1_encode_sr(float(v), int(r16))


def e4m3_decode(code: int) -> float:
    return lib().bsqo_e4m3_decode(int(code))


def e4m3_encode(v: float) -> int:
    return lib().bsqo_e4m3_encode(float(v))


def e4m3_encode_sr(v: float, r16: int) -> int:
    return lib().bsqo_e4m3_encode_sr(float(v), int(r16))


def e8m0_decode(code: int) -> float:
    return lib().bsqo_e8m0_decode(int(code))


def e2m1_encode_array(v: np.ndarray) -> np.ndarray:
    v = _c(v, np.float32).ravel()
    out = np.empty(v.size, np.uint8)
    lib().bsqo_e2m1_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    v = _c(v, np.float32).ravel()
    out = np.empty(v.size, np.uint8)
    lib().bsqo_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


# ---------------------------------------------------------------- philox
def philox4x32_10(ctr, key) -> np.ndarray:
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.empty(4, np.uint32)
    lib().bsqo_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def sr_bits16(seed: int, stream: int, idx: int) -> int:
    return lib().bsqo_sr_bits16(int(seed), int(stream), int(idx))


# ---------------------------------------------------------------- NVFP4
def nvfp4_quantize_rows(x_bits: np.ndarray, four_six: bool = False):
    """Per-row (per-token) NVFP4 quantization of a bf16 [rows, K] tensor.
    Returns (codes [rows, K/2] u8, sf [rows, K/16] u8 linear, t [rows] f32)."""
    x = _c(x_bits, np.uint16)
    rows, K = x.shape
    codes = np.empty((rows, K // 2), np.uint8)
    sf = np.empty((rows, K // 16), np.uint8)
    t = np.empty(rows, np.float32)
    lib().bsqo_nvfp4_quantize_rows(_ptr(x), rows, K, K, int(four_six), _ptr(codes), _ptr(sf), _ptr(t))
    return codes, sf, t


def nvfp4_quantize_rows_given_t(x: np.ndarray, t: np.ndarray, four_six: bool = False):
    """NVFP4 quantization of binary32 rows with caller-supplied row scales."""
    x = _c(x, np.float32)
    rows, K = x.shape
    t = _c(t, np.float32)
    codes = np.empty((rows, K // 2), np.uint8)
    sf = np.empty((rows, K // 16), np.uint8)
    lib().bsqo_nvfp4_quantize_rows_given_t(_ptr(x), rows, K, _ptr(t), int(four_six), _ptr(codes), _ptr(sf))
    return codes, sf


def nvfp4_quantize_group(x_bits: np.ndarray):
    """One FP32 scale per group: x is bf16 [groups, rows, K] (weights)."""
    x = _c(x_bits, np.uint16)
    G, rows, K = x.shape
    codes = np.empty((G, rows, K // 2), np.uint8)
    sf = np.empty((G, rows, K // 16), np.uint8)
    t = np.empty(G, np.float32)
    lib().bsqo_nvfp4_quantize_group(_ptr(x), G, rows, K, _ptr(codes), _ptr(sf), _ptr(t))
    return codes, sf, t


def nvfp4_block_candidate(x16: np.ndarray, t: float, mult: float):
    """One candidate (block-scale multiplier 6 or 4) of a 16-value block:
    returns (unpacked codes [16], SF byte, fp32 tree-summed SSE)."""
    x = _c(x16, np.float32)
    codes = np.empty(16, np.uint8)
    sf = np.empty(1, np.uint8)
    sse = np.empty(1, np.float32)
    lib().bsqo_nvfp4_block_candidate(_ptr(x), float(t), float(mult), _ptr(codes), _ptr(sf), _ptr(sse))
    return codes, int(sf[0]), float(sse[0])


def nvfp4_dequantize(codes, sf, t) -> np.ndarray:
    codes = _c(codes, np.uint8)
    sf = _c(sf, np.uint8)
    t = _c(t, np.float32)
    rows = codes.shape[0]
    K = codes.shape[1] * 2
    out = np.empty((rows, K), np.float32)
    lib().bsqo_nvfp4_dequantize(_ptr(codes), _ptr(sf), _ptr(t), rows, K, _ptr(out))
    return out


def nvfp4_quantize_2d(x_bits: np.ndarray):
    """2-D NVFP4 of bf16 x [rows, K]: one E4M3 scale per 16 x 16 tile and one
    FP32 scale per tensor ("End-to-End 4-Bit Training", section "第二个决定": square
    block scales are the same before and after the transpose).  Returns
    (codes [rows, K/2], tile scales [rows/16, K/16], t)."""
    x = _c(x_bits, np.uint16)
    rows, K = x.shape
    codes = np.empty((rows, K // 2), np.uint8)
    sf = np.empty((rows // 16, K // 16), np.uint8)
    t = np.empty(1, np.float32)
    lib().bsqo_nvfp4_quantize_2d(_ptr(x), rows, K, _ptr(codes), _ptr(sf), _ptr(t))
    return codes, sf, float(t[0])


def rht_signs(seed: int) -> int:
    """The 32 signs of the random Hadamard transform as a bit mask (bit j set:
    s_j = -1), from Philox4x32-10 stream 2."""
    return int(lib().bsqo_rht_signs(int(seed)))


def rht32(x: np.ndarray, signs: int) -> np.ndarray:
    """y = H32 (s . x) per 32-element group of the last axis, binary32 in the
    butterfly order ("End-to-End 4-Bit Training", section "第三个决定")."""
    xf = _c(x, np.float32)
    y = np.empty_like(xf)
    lib().bsqo_rht32(_ptr(xf), xf.size, int(signs), _ptr(y))
    return y


def nvfp4_quantize_rht(x_bits: np.ndarray, seed: int):
    """Per-token NVFP4 of the 32-point random Hadamard transform of bf16 x
    [rows, K] (K % 32 == 0): (codes [rows, K/2], sf [rows, K/16], t [rows])."""
    x = _c(x_bits, np.uint16)
    rows, K = x.shape
    codes = np.empty((rows, K // 2), np.uint8)
    sf = np.empty((rows, K // 16), np.uint8)
    t = np.empty(rows, np.float32)
    lib().bsqo_nvfp4_quantize_rht(_ptr(x), rows, K, int(seed), _ptr(codes), _ptr(sf), _ptr(t))
    return codes, sf, t


def nvfp4_dequantize_bf16(codes, sf, t_rows) -> np.ndarray:
    """The BF16 operands of the dequantized backward mode ("LMSYS Drops Miles
    ...", section "Recipe 2: Per-token NVFP4 for MoE experts": backward GEMMs
    run in BF16 on BF16 dequantizations of the exact low-precision forward
    operands).  The binary32 dequantization of the per-row recipe (element
    value times its block scale, then times the row's FP32 scale, one
    rounding per product), rounded to bf16 to nearest with ties to even.
    READING: the pages fix no rounding for this step; BF16 round-to-nearest
    of the binary32 value is the plainest.  t_rows: one scale per row (a
    per-expert scale is repeated over its rows).  Returns uint16 bf16 bits."""
    d = nvfp4_dequantize(codes, sf, t_rows)
    return f64_to_bf16_array(d.astype(np.float64))


def sf_swizzled_offset(row: int, kblock: int, K: int) -> int:
    return lib().bsqo_sf_swizzled_offset(int(row), int(kblock), int(K))


def sf_to_swizzled(sf_linear: np.ndarray) -> np.ndarray:
    """Place a linear SF matrix [rows, cols] into the tensor-core layout
    (rows padded to 128, columns to 4; padding bytes are 0)."""
    sf_linear = _c(sf_linear, np.uint8)
    rows, cols = sf_linear.shape
    out = np.empty(((rows + 127) // 128 * 128) * ((cols + 3) // 4 * 4), np.uint8)
    lib().bsqo_sf_swizzle(_ptr(sf_linear), rows, cols, _ptr(out))
    return out


# ---------------------------------------------------------------- MXFP8
def mxfp8_quantize_rowcol(x_bits: np.ndarray, row: bool = True, col: bool = True):
    """MXFP8 quantization of bf16 [rows, K]: row copy (codes [rows, K], SF
    [rows, K/32]) and column copy stored transposed (codes [K, rows], SF
    [K, rows/32])."""
    x = _c(x_bits, np.uint16)
    rows, K = x.shape
    rc = np.empty((rows, K), np.uint8) if row else None
    rs = np.empty((rows, K // 32), np.uint8) if row else None
    cc = np.empty((K, rows), np.uint8) if col else None
    cs = np.empty((K, rows // 32), np.uint8) if col else None
    lib().bsqo_mxfp8_quantize_rowcol(_ptr(x), rows, K, K, _ptr(rc), _ptr(rs), _ptr(cc), _ptr(cs))
    return rc, rs, cc, cs


# ---------------------------------------------------------------- requant
def requant_transpose(codes, sf, t, sr: bool, seed: int, nvfp4: bool = True, mxfp8: bool = True):
    """Dequantize an NVFP4 [rows, K] tensor, transpose, requantize to NVFP4
    (codes [K, rows/2], SF [K, rows/16], t [K]) and/or MXFP8 (codes [K, rows],
    SF [K, rows/32]); RNE, or stochastic rounding with Philox bits."""
    codes = _c(codes, np.uint8)
    sf = _c(sf, np.uint8)
    t = _c(t, np.float32)
    M = codes.shape[0]
    K = codes.shape[1] * 2
    nc = np.empty((K, M // 2), np.uint8) if nvfp4 else None
    ns = np.empty((K, M // 16), np.uint8) if nvfp4 else None
    nt = np.empty(K, np.float32) if nvfp4 else None
    mc = np.empty((K, M), np.uint8) if mxfp8 else None
    ms = np.empty((K, M // 32), np.uint8) if mxfp8 else None
    lib().bsqo_requant_transpose(_ptr(codes), _ptr(sf), _ptr(t), M, K, int(sr), int(seed),
                                 _ptr(nc), _ptr(ns), _ptr(nt), _ptr(mc), _ptr(ms))
    return nc, ns, nt, mc, ms


# ---------------------------------------------------------------- GEMM
def gemm_nvfp4(a_codes, a_sf, a_t, b_codes, b_sf, b_t: float, with_abs: bool = True):
    """fp64 GEMM on exactly dequantized NVFP4 operands: out[m, n] =
    sum_k A[m, k] * B[n, k]. Returns (out, sum_k |A*B|)."""
    a_codes = _c(a_codes, np.uint8)
    a_sf = _c(a_sf, np.uint8)
    a_t = _c(a_t, np.float32)
    b_codes = _c(b_codes, np.uint8)
    b_sf = _c(b_sf, np.uint8)
    M = a_codes.shape[0]
    K = a_codes.shape[1] * 2
    N = b_codes.shape[0]
    out = np.empty((M, N), np.float64)
    ab = np.empty((M, N), np.float64) if with_abs else None
    lib().bsqo_gemm_nvfp4(_ptr(a_codes), _ptr(a_sf), _ptr(a_t), M, K, _ptr(b_codes), _ptr(b_sf),
                          float(b_t), N, _ptr(out), _ptr(ab))
    return out, ab


def gemm_mxfp8(a_codes, a_sf, a_t, b_codes, b_sf, b_t: float = 1.0, with_abs: bool = True):
    """fp64 GEMM on exactly dequantized MXFP8 operands (codes [rows, K] E4M3,
    SF [rows, K/32] E8M0 linear): out[m, n] = sum_k A[m, k] * B[n, k].
    Returns (out, sum_k |A*B|)."""
    a_codes = _c(a_codes, np.uint8)
    a_sf = _c(a_sf, np.uint8)
    a_t = _c(a_t, np.float32)
    b_codes = _c(b_codes, np.uint8)
    b_sf = _c(b_sf, np.uint8)
    M, K = a_codes.shape
    N = b_codes.shape[0]
    out = np.empty((M, N), np.float64)
    ab = np.empty((M, N), np.float64) if with_abs else None
    lib().bsqo_gemm_mxfp8(_ptr(a_codes), _ptr(a_sf), _ptr(a_t), M, K, _ptr(b_codes), _ptr(b_sf), float(b_t), N,
                          _ptr(out), _ptr(ab))
    return out, ab


def gemm_nvfp4_sampled(a_codes, a_sf, a_t, b_codes, b_sf, b_t, a_rows, b_rows, b_group):
    """Selected output elements: sample s is row a_rows[s] of A against row
    b_rows[s] of B (all groups' rows stacked), B scale b_t[b_group[s]]."""
    a_codes = _c(a_codes, np.uint8)
    a_sf = _c(a_sf, np.uint8)
    a_t = _c(a_t, np.float32)
    b_codes = _c(b_codes, np.uint8)
    b_sf = _c(b_sf, np.uint8)
    b_t = _c(b_t, np.float32)
    ar = _c(a_rows, np.int64)
    br = _c(b_rows, np.int64)
    bg = _c(b_group, np.int64)
    K = a_codes.shape[-1] * 2
    out = np.empty(ar.size, np.float64)
    ab = np.empty(ar.size, np.float64)
    lib().bsqo_gemm_nvfp4_sampled(_ptr(a_codes), _ptr(a_sf), _ptr(a_t), K, _ptr(b_codes), _ptr(b_sf),
                                  _ptr(b_t), _ptr(ar), _ptr(br), _ptr(bg), ar.size, _ptr(out), _ptr(ab))
    return out, ab


# ---------------------------------------------------------------- MoE pieces
def route(topk_ids: np.ndarray, E: int, pad: int = 128):
    """Returns (offsets [E+1], slot_of [T*k], row_src [R_pad])."""
    ids = _c(topk_ids, np.int32)
    T, k = ids.shape
    offsets = np.empty(E + 1, np.int32)
    slot_of = np.empty(T * k, np.int32)
    cap = T * k + E * (pad - 1)
    row_src = np.empty(cap, np.int32)
    rpad = lib().bsqo_route(_ptr(ids), T, k, E, pad, _ptr(offsets), _ptr(slot_of), _ptr(row_src))
    return offsets, slot_of, row_src[:rpad].copy()


def swiglu(gate_up: np.ndarray) -> np.ndarray:
    gu = _c(gate_up, np.float64)
    rows, twoI = gu.shape
    h = np.empty((rows, twoI // 2), np.float64)
    lib().bsqo_swiglu(_ptr(gu), rows, twoI // 2, _ptr(h))
    return h


def combine(out_rows_bits: np.ndarray, slot_of: np.ndarray, topk_w: np.ndarray) -> np.ndarray:
    o = _c(out_rows_bits, np.uint16)
    H = o.shape[1]
    s = _c(slot_of, np.int32)
    w = _c(topk_w, np.float32)
    T, k = w.shape
    y = np.empty((T, H), np.uint16)
    lib().bsqo_combine(_ptr(o), H, _ptr(s), _ptr(w), T, k, _ptr(y))
    return y


def f64_to_bf16(v: float) -> int:
    return lib().bsqo_f64_to_bf16(float(v))


def f64_to_bf16_array(v: np.ndarray) -> np.ndarray:
    flat = _c(v, np.float64).ravel()
    out = np.empty(flat.size, np.uint16)
    lib().bsqo_f64_to_bf16_array(_ptr(flat), flat.size, _ptr(out))
    return out.reshape(np.shape(v))
