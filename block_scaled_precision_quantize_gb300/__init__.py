"""Block-scaled (NVFP4 / MXFP8) quantization and grouped expert GEMM for
GB300 -- Python binding of the C ABI in include/bsq.h.

The functions here only marshal arguments: they allocate output tensors with
PyTorch on the input's device, pass raw device pointers and the current CUDA
stream to libbsq.so, and raise on a non-OK status. Every step of the
computation runs in the library's CUDA kernels; there is no CPU fallback, and
loading fails loudly if the library has not been built (``build()``).
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "load", "build", "BsqError",
    "quantize_nvfp4_per_token", "quantize_nvfp4_per_expert", "quantize_mxfp8_rowcol",
    "quantize_nvfp4_2d", "quantize_nvfp4_rht", "dequantize_nvfp4", "requant_transpose_sr",
    "grouped_expert_gemm_fp4", "grouped_expert_gemm_mxfp8", "moe_expert_forward",
    "moe_workspace_layout", "moe_workspace_size", "requant_workspace_size",
    "sf_swizzle", "sf_unswizzle", "format_probe", "philox_bits16", "sf_swizzled_bytes", "mma_ceiling",
    "check_status",
    "SF_SWIZZLED", "FOUR_SIX", "STOCHASTIC", "MOE_FUSED_H", "MOE_KEEP_H", "EPI_F32", "EPI_BF16", "EPI_SWIGLU_BF16",
]

SF_SWIZZLED = 1 << 0
FOUR_SIX = 1 << 1
STOCHASTIC = 1 << 2
MOE_FUSED_H = 1 << 3
MOE_KEEP_H = 1 << 4
EPI_F32, EPI_BF16, EPI_SWIGLU_BF16 = 0, 1, 2
DEV_OK, DEV_TIMEOUT, DEV_BAD_OFFSETS, DEV_BAD_EXPERT = 0, 1, 2, 3

_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64
_U32 = ctypes.c_uint32
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t


class BsqError(RuntimeError):
    pass


class MoeLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "offsets", "counts", "slot_of", "row_src", "xq_codes", "xq_sf", "xq_scale", "h",
        "hq_codes", "hq_sf", "hq_scale", "out", "scan", "h_scratch", "total")] + [("capacity", ctypes.c_int64)]


_SIGS = {
    "bsq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "bsq_version": (_I32, []),
    "bsq_check_status": (ctypes.c_int, [_P, ctypes.POINTER(_I32), _P]),
    "quantize_nvfp4_per_token": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _P, _U32, _P, _P]),
    "quantize_nvfp4_per_expert": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _P, _U32, _P, _P]),
    "quantize_mxfp8_rowcol": (ctypes.c_int, [_P, _I64, _I64, _I64, _P, _P, _P, _P, _U32, _P, _P]),
    "dequantize_nvfp4": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I64, _P, _I64, _U32, _P, _P]),
    "quantize_nvfp4_2d": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P, _P, _P, _U32, _P, _P]),
    "quantize_nvfp4_rht": (ctypes.c_int, [_P, _I64, _I64, _I64, _U64, _P, _P, _P, _U32, _P, _P]),
    "bsq_requant_workspace_size": (_SZ, [_I64, _I64, _I32]),
    "requant_transpose_sr": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _P, _P, _P, _P, _P, _U64, _P, _SZ, _U32,
                                            _P, _P]),
    "grouped_expert_gemm_fp4": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _I32, _P,
                                               _I64, _U32, _P, _P]),
    "grouped_expert_gemm_mxfp8": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P, _I32, _P,
                                                 _I64, _U32, _P, _P]),
    "bsq_moe_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, _I64]),
    "bsq_moe_workspace_layout": (ctypes.c_int, [_I64, _I64, _I64, _I64, _I64, ctypes.POINTER(MoeLayout)]),
    "moe_expert_forward": (ctypes.c_int, [_P, _I64, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                          _P, _SZ, _U32, _P, _P]),
    "bsq_sf_swizzle": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
    "bsq_sf_unswizzle": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
    "bsq_format_probe": (ctypes.c_int, [_I32, _P, _P, _P, _I64, _P]),
    "bsq_philox_bits16": (ctypes.c_int, [_U64, _U32, _U64, _I64, _P, _P]),
    "bsq_set_stage_events": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), _I32]),
    "bsq_mma_ceiling": (ctypes.c_int, [_I32, _I32, _I32, _P, ctypes.POINTER(_I32), _P, _P]),
}

_stage_array = None


def set_stage_events(events):
    """Profiling hook: moe_expert_forward records the 7 given torch.cuda.Event
    objects at its stage boundaries (None clears). Events must have been
    recorded once so that their CUDA handles exist."""
    global _stage_array
    if events is None:
        _stage_array = None
        _check(load().bsq_set_stage_events(None, 0), "bsq_set_stage_events")
        return
    if any(not e.cuda_event for e in events):
        raise ValueError("set_stage_events: record each event once first (torch creates the CUDA event lazily)")
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _stage_array = arr  # keep alive while set
    _check(load().bsq_set_stage_events(arr, len(events)), "bsq_set_stage_events")


def build(force: bool = False) -> str:
    """Compile libbsq.so for sm_103a (nvcc; no GPU needed)."""
    return _build.build(force=force)


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libbsq.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise BsqError(f"CUDA library not built: {path} is missing (run build())")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int, what: str):
    if status != 0:
        msg = load().bsq_status_string(status).decode()
        raise BsqError(f"{what}: {msg} (status {status})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def check_status(dev_status) -> int:
    """The device status word `dev_status` (int32 CUDA tensor) read back on
    the current stream after the work enqueued there (bsq_check_status:
    waits for the stream).  Returns DEV_OK or the first DEV_* recorded."""
    _cuda(dev_status, "dev_status")
    out = _I32(0)
    _check(load().bsq_check_status(_ptr(dev_status), ctypes.byref(out), _stream(dev_status.device)),
           "bsq_check_status")
    return int(out.value)


def _cuda(t, name):
    if not t.is_cuda:
        raise BsqError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise BsqError(f"{name} must be contiguous")


def sf_swizzled_bytes(rows: int, cols: int) -> int:
    """Size of a swizzled SF buffer for an SF matrix [rows][cols]."""
    return ((rows + 127) // 128 * 128) * ((cols + 3) // 4 * 4)


def _sf_alloc(rows, cols, swizzled, device, lead=()):
    if swizzled:
        return torch.empty(sf_swizzled_bytes(rows, cols), dtype=torch.uint8, device=device)
    return torch.empty(*lead, rows, cols, dtype=torch.uint8, device=device)


# ---------------------------------------------------------------- quantizers
def quantize_nvfp4_per_token(x, four_six=False, swizzled=False, dev_status=None):
    """Per-token NVFP4 of bf16 x [rows, K]: (codes [rows, K/2] u8, sf u8,
    row_scale [rows] f32)."""
    _cuda(x, "x")
    rows, K = x.shape
    codes = torch.empty(rows, K // 2, dtype=torch.uint8, device=x.device)
    sf = _sf_alloc(rows, K // 16, swizzled, x.device)
    scale = torch.empty(rows, dtype=torch.float32, device=x.device)
    flags = (SF_SWIZZLED if swizzled else 0) | (FOUR_SIX if four_six else 0)
    _check(load().quantize_nvfp4_per_token(_ptr(x), rows, K, K, _ptr(codes), _ptr(sf), _ptr(scale), flags,
                                           _ptr(dev_status), _stream(x.device)), "quantize_nvfp4_per_token")
    return codes, sf, scale


def quantize_nvfp4_per_expert(w, swizzled=True, dev_status=None):
    """NVFP4 weights bf16 [E, rows, K] with one FP32 scale per expert."""
    _cuda(w, "w")
    E, rows, K = w.shape
    codes = torch.empty(E, rows, K // 2, dtype=torch.uint8, device=w.device)
    sf = _sf_alloc(E * rows, K // 16, swizzled, w.device)
    if not swizzled:
        sf = sf.view(E, rows, K // 16)
    scale = torch.empty(E, dtype=torch.float32, device=w.device)
    _check(load().quantize_nvfp4_per_expert(_ptr(w), E, rows, K, _ptr(codes), _ptr(sf), _ptr(scale),
                                            SF_SWIZZLED if swizzled else 0, _ptr(dev_status), _stream(w.device)),
           "quantize_nvfp4_per_expert")
    return codes, sf, scale


def quantize_mxfp8_rowcol(x, row=True, col=True, swizzled=False, dev_status=None):
    """MXFP8 copies of bf16 x [rows, K]: (row_codes [rows, K], row_sf,
    col_codes [K, rows], col_sf); a skipped copy is returned as None."""
    _cuda(x, "x")
    rows, K = x.shape
    dev = x.device
    rc = torch.empty(rows, K, dtype=torch.uint8, device=dev) if row else None
    rs = _sf_alloc(rows, K // 32, swizzled, dev) if row else None
    cc = torch.empty(K, rows, dtype=torch.uint8, device=dev) if col else None
    cs = _sf_alloc(K, rows // 32, swizzled, dev) if col else None
    _check(load().quantize_mxfp8_rowcol(_ptr(x), rows, K, K, _ptr(rc), _ptr(rs), _ptr(cc), _ptr(cs),
                                        SF_SWIZZLED if swizzled else 0, _ptr(dev_status), _stream(dev)),
           "quantize_mxfp8_rowcol")
    return rc, rs, cc, cs


def quantize_nvfp4_rht(x, seed=0, swizzled=False, dev_status=None):
    """Per-token NVFP4 of the 32-point random Hadamard transform of each row of
    bf16 x [rows, K] (K % 32 == 0): (codes [rows, K/2], sf, row_scale [rows])."""
    _cuda(x, "x")
    rows, K = x.shape
    codes = torch.empty(rows, K // 2, dtype=torch.uint8, device=x.device)
    sf = _sf_alloc(rows, K // 16, swizzled, x.device)
    scale = torch.empty(rows, dtype=torch.float32, device=x.device)
    _check(load().quantize_nvfp4_rht(_ptr(x), rows, K, K, int(seed), _ptr(codes), _ptr(sf), _ptr(scale),
                                     SF_SWIZZLED if swizzled else 0, _ptr(dev_status), _stream(x.device)),
           "quantize_nvfp4_rht")
    return codes, sf, scale


def quantize_nvfp4_2d(x, transposed=True, dev_status=None):
    """2-D NVFP4 of bf16 x [rows, K] (rows % 16 == 0): one E4M3 scale per
    16 x 16 tile and one FP32 scale per tensor.  Returns (codes [rows, K/2],
    tile scales [rows/16, K/16], codes of x^T [K, rows/2], tile scales of x^T
    [K/16, rows/16], tensor scale [1]); the transposed pair is None when
    `transposed` is False."""
    _cuda(x, "x")
    rows, K = x.shape
    dev = x.device
    codes = torch.empty(rows, K // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty(rows // 16, K // 16, dtype=torch.uint8, device=dev)
    codes_t = torch.empty(K, rows // 2, dtype=torch.uint8, device=dev) if transposed else None
    sf_t = torch.empty(K // 16, rows // 16, dtype=torch.uint8, device=dev) if transposed else None
    scale = torch.zeros(1, dtype=torch.float32, device=dev)
    _check(load().quantize_nvfp4_2d(_ptr(x), rows, K, _ptr(codes), _ptr(sf), _ptr(codes_t), _ptr(sf_t), _ptr(scale),
                                    0, _ptr(dev_status), _stream(dev)), "quantize_nvfp4_2d")
    return codes, sf, codes_t, sf_t, scale


def dequantize_nvfp4(codes, sf, scale, swizzled=False, y=None, dev_status=None):
    """BF16 dequantization of NVFP4 codes [..., K/2] (the operands of the
    dequantized backward).  `scale` holds one FP32 scale per row (per-token)
    or per group of rows (per-expert weights [E, N, K/2] with scale [E]);
    returns bf16 [..., K] (or writes `y`, rows of pitch y.stride(-2))."""
    _cuda(codes, "codes")
    _cuda(sf, "sf")
    _cuda(scale, "scale")
    K = 2 * codes.shape[-1]
    rows = codes.numel() // codes.shape[-1] if codes.numel() else 0
    groups = scale.numel()
    if rows and (groups == 0 or rows % groups != 0):
        raise BsqError(f"dequantize_nvfp4: {groups} scales for {rows} rows")
    if y is None:
        y = torch.empty(*codes.shape[:-1], K, dtype=torch.bfloat16, device=codes.device)
    elif not (y.is_cuda and y.dtype == torch.bfloat16 and y.dim() == 2 and y.shape == (rows, K) and y.stride(-1) == 1):
        raise BsqError("dequantize_nvfp4: y must be a CUDA bf16 [rows, K] tensor with unit column stride")
    ldy = y.stride(-2) if y.dim() >= 2 else K
    _check(load().dequantize_nvfp4(_ptr(codes), _ptr(sf), _ptr(scale), rows, K, rows // groups if rows else 1,
                                   _ptr(y), ldy, SF_SWIZZLED if swizzled else 0, _ptr(dev_status),
                                   _stream(codes.device)), "dequantize_nvfp4")
    return y


def requant_workspace_size(rows, K, nvfp4=True) -> int:
    return load().bsq_requant_workspace_size(rows, K, 1 if nvfp4 else 0)


def requant_transpose_sr(codes, sf, scale, nvfp4=True, mxfp8=True, stochastic=True, seed=0, swizzled=False,
                         workspace=None, out=None, dev_status=None):
    """Dequantize NVFP4 [rows, K] (codes [rows, K/2]), transpose, requantize
    to NVFP4 and/or MXFP8 with RNE or Philox stochastic rounding.
    Returns dict nv_codes [K, rows/2], nv_sf, nv_scale [K], mx_codes [K, rows],
    mx_sf (absent targets are None). `out` may hold preallocated tensors."""
    _cuda(codes, "codes")
    rows, K = codes.shape[0], codes.shape[1] * 2
    dev = codes.device
    o = dict(out or {})
    if nvfp4:
        o.setdefault("nv_codes", torch.empty(K, rows // 2, dtype=torch.uint8, device=dev))
        o.setdefault("nv_sf", _sf_alloc(K, rows // 16, swizzled, dev))
        o.setdefault("nv_scale", torch.empty(K, dtype=torch.float32, device=dev))
    if mxfp8:
        o.setdefault("mx_codes", torch.empty(K, rows, dtype=torch.uint8, device=dev))
        o.setdefault("mx_sf", _sf_alloc(K, rows // 32, swizzled, dev))
    need = requant_workspace_size(rows, K, nvfp4)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    flags = (SF_SWIZZLED if swizzled else 0) | (STOCHASTIC if stochastic else 0)
    g = o.get
    _check(load().requant_transpose_sr(
        _ptr(codes), _ptr(sf), _ptr(scale), rows, K,
        _ptr(g("nv_codes")) if nvfp4 else None, _ptr(g("nv_sf")) if nvfp4 else None,
        _ptr(g("nv_scale")) if nvfp4 else None,
        _ptr(g("mx_codes")) if mxfp8 else None, _ptr(g("mx_sf")) if mxfp8 else None,
        int(seed), _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
        flags, _ptr(dev_status), _stream(dev)), "requant_transpose_sr")
    for k in ("nv_codes", "nv_sf", "nv_scale", "mx_codes", "mx_sf"):
        o.setdefault(k, None)
    return o


# ---------------------------------------------------------------- GEMM
def grouped_expert_gemm_fp4(a_codes, a_sf, a_scale, offsets, b_codes, b_sf, b_scale, epilogue=EPI_F32,
                            out=None, dev_status=None):
    """Grouped block-scaled GEMM. a_codes [M, K/2] (expert-sorted rows,
    segments given by int32 offsets [E+1], multiples of 128), b_codes
    [E, N, K/2]; SF swizzled. Returns out ([M, N] fp32/bf16 or [M, N/2] bf16
    for SwiGLU)."""
    for t, n in ((a_codes, "a_codes"), (b_codes, "b_codes"), (offsets, "offsets")):
        _cuda(t, n)
    M, K = a_codes.shape[0], a_codes.shape[1] * 2
    E, N = b_codes.shape[0], b_codes.shape[1]
    ncols = N // 2 if epilogue == EPI_SWIGLU_BF16 else N
    dt = torch.float32 if epilogue == EPI_F32 else torch.bfloat16
    if out is None:
        out = torch.empty(M, ncols, dtype=dt, device=a_codes.device)
    _check(load().grouped_expert_gemm_fp4(_ptr(a_codes), _ptr(a_sf), _ptr(a_scale), _ptr(offsets), E, M, K, N,
                                          _ptr(b_codes), _ptr(b_sf), _ptr(b_scale), epilogue, _ptr(out),
                                          out.stride(0), SF_SWIZZLED, _ptr(dev_status), _stream(a_codes.device)),
           "grouped_expert_gemm_fp4")
    return out


def grouped_expert_gemm_mxfp8(a_codes, a_sf, offsets, b_codes, b_sf, a_scale=None, b_scale=None,
                              epilogue=EPI_F32, out=None, dev_status=None):
    """Grouped block-scaled GEMM on MXFP8 operands: a_codes [M, K] E4M3
    (expert-sorted rows, segments given by int32 offsets [E+1], multiples of
    128), b_codes [E, N, K]; E8M0 SF swizzled.  a_scale [M] / b_scale [E]
    default to ones.  Returns out [M, N] (fp32 or bf16)."""
    for t, n in ((a_codes, "a_codes"), (b_codes, "b_codes"), (offsets, "offsets")):
        _cuda(t, n)
    M, K = a_codes.shape
    E, N = b_codes.shape[0], b_codes.shape[1]
    dev = a_codes.device
    if a_scale is None:
        a_scale = torch.ones(M, dtype=torch.float32, device=dev)
    if b_scale is None:
        b_scale = torch.ones(E, dtype=torch.float32, device=dev)
    dt = torch.float32 if epilogue == EPI_F32 else torch.bfloat16
    if out is None:
        out = torch.empty(M, N, dtype=dt, device=dev)
    _check(load().grouped_expert_gemm_mxfp8(_ptr(a_codes), _ptr(a_sf), _ptr(a_scale), _ptr(offsets), E, M, K, N,
                                            _ptr(b_codes), _ptr(b_sf), _ptr(b_scale), epilogue, _ptr(out),
                                            out.stride(0), SF_SWIZZLED, _ptr(dev_status), _stream(dev)),
           "grouped_expert_gemm_mxfp8")
    return out


# ---------------------------------------------------------------- MoE
def moe_workspace_layout(T, H, I, E, topk) -> MoeLayout:
    L = MoeLayout()
    _check(load().bsq_moe_workspace_layout(T, H, I, E, topk, ctypes.byref(L)), "bsq_moe_workspace_layout")
    return L


def moe_workspace_size(T, H, I, E, topk) -> int:
    return int(load().bsq_moe_workspace_size(T, H, I, E, topk))


def moe_expert_forward(x, topk_ids, topk_weights, wgu, wd, I, four_six=False, workspace=None, y=None,
                       dev_status=None, fused_h=False, keep_h=False):
    """Routed SwiGLU experts with NVFP4 activations/weights. x bf16 [T, H];
    topk_ids int32 [T, k]; topk_weights f32 [T, k]; wgu = (codes [E, 2I, H/2],
    sf, scale [E]); wd = (codes [E, H, I/2], sf, scale [E]). Returns y bf16
    [T, H]; pass `workspace` (uint8, moe_workspace_size bytes) to keep the
    intermediates.  fused_h=True quantizes h inside GEMM1's epilogue (same
    results); with it, keep_h=True also keeps the bf16 h in the workspace."""
    _cuda(x, "x")
    T, H = x.shape
    k = topk_ids.shape[1]
    E = wgu[0].shape[0]
    dev = x.device
    if workspace is None:
        workspace = torch.empty(moe_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=dev)
    if y is None:
        y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    _check(load().moe_expert_forward(_ptr(x), T, H, I, E, k, _ptr(topk_ids), _ptr(topk_weights),
                                     _ptr(wgu[0]), _ptr(wgu[1]), _ptr(wgu[2]), _ptr(wd[0]), _ptr(wd[1]),
                                     _ptr(wd[2]), _ptr(y), _ptr(workspace), workspace.numel(),
                                     (FOUR_SIX if four_six else 0) | (MOE_FUSED_H if fused_h else 0) |
                                     (MOE_KEEP_H if keep_h else 0),
                                     _ptr(dev_status), _stream(dev)),
           "moe_expert_forward")
    return y


# ---------------------------------------------------------------- helpers
def sf_swizzle(sf_linear):
    _cuda(sf_linear, "sf_linear")
    rows, cols = sf_linear.shape
    out = torch.empty(sf_swizzled_bytes(rows, cols), dtype=torch.uint8, device=sf_linear.device)
    _check(load().bsq_sf_swizzle(_ptr(sf_linear), rows, cols, _ptr(out), _stream(out.device)), "bsq_sf_swizzle")
    return out


def sf_unswizzle(sf_swz, rows, cols):
    _cuda(sf_swz, "sf_swizzled")
    out = torch.empty(rows, cols, dtype=torch.uint8, device=sf_swz.device)
    _check(load().bsq_sf_unswizzle(_ptr(sf_swz), rows, cols, _ptr(out), _stream(out.device)), "bsq_sf_unswizzle")
    return out


def format_probe(kind, values, rbits=None):
    """Run the kernels' own element conversions on a float32 CUDA tensor."""
    _cuda(values, "values")
    n = values.numel()
    dt = torch.uint8 if kind < 4 else torch.float32
    out = torch.empty(n, dtype=dt, device=values.device)
    _check(load().bsq_format_probe(kind, _ptr(values), _ptr(rbits), _ptr(out), n, _stream(values.device)),
           "bsq_format_probe")
    return out


def mma_ceiling(fmt, cta_group, iters, device="cuda", dev_status=None):
    """Launch the MMA-ceiling kernel once (fmt 0 NVFP4 / 1 MXFP8, cta_group 1
    or 2, `iters` MMAs per CTA) on the current stream.  Returns (ctas,
    cycles): the CTAs launched and a device uint64 tensor of per-CTA cycle
    counts (0 for the second CTA of a pair)."""
    props = torch.cuda.get_device_properties(device)
    cycles = torch.zeros(props.multi_processor_count, dtype=torch.int64, device=device)
    ctas = _I32(0)
    _check(load().bsq_mma_ceiling(int(fmt), int(cta_group), int(iters), _ptr(cycles), ctypes.byref(ctas),
                                  _ptr(dev_status), _stream(cycles.device)), "bsq_mma_ceiling")
    return ctas.value, cycles


def philox_bits16(seed, stream_id, idx0, n, device="cuda"):
    out = torch.empty(n, dtype=torch.int16, device=device)
    _check(load().bsq_philox_bits16(int(seed), int(stream_id), int(idx0), n, _ptr(out), _stream(out.device)),
           "bsq_philox_bits16")
    return out
