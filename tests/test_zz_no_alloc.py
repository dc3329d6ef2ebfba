"""requant_transpose_sr_noalloc: the allocation-free entry point for callers
that cannot give the library device scratch memory (a host framework that
owns only its input and output buffers, or code that must not allocate
device memory once running).  It keeps the column maxima in a fixed array
inside the library, so it takes no workspace; its results must equal those of
requant_transpose_sr and of the oracle.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test."""
import ctypes
import os
import shutil

import numpy as np
import pytest
import torch

from block_scaled_precision_quantize_gb300 import synth
from conftest import bits_equal, first_mismatch, guarded_empty, to_dev, to_np

P = ctypes.c_void_p
I64 = ctypes.c_int64
ARGTYPES = [P, P, P, I64, I64, P, P, P, P, P, ctypes.c_uint64, ctypes.c_uint32, P, P]


def _fn():
    import block_scaled_precision_quantize_gb300 as bsq
    bsq.build()
    fn = bsq.load().requant_transpose_sr_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = ARGTYPES
    return bsq, fn


def _have_library():
    import block_scaled_precision_quantize_gb300 as bsq
    return os.path.exists(bsq.lib_path()) or shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")


def test_noalloc_rejects_k_beyond_its_array():
    """Host-side checks only (nothing is enqueued): K past the fixed array and
    unknown flags are refused before the device is touched."""
    if not _have_library():
        pytest.skip("the CUDA library is not built and nvcc is not available to build it")
    _, fn = _fn()
    d = P(4096)
    assert fn(d, d, d, 64, 65536 + 16, d, d, d, None, None, 0, 0, None, None) == 2  # BSQ_ERR_SHAPE
    assert fn(d, d, d, 64, 96, d, d, d, None, None, 0, 1 << 9, None, None) == 4     # BSQ_ERR_FLAGS


def _call(bsq, fn, codes, sf, t, rows, K, out, seed, sr, swz):
    g = out.get
    st = fn(P(codes.data_ptr()), P(sf.data_ptr()), P(t.data_ptr()), rows, K,
            P(g("nv_codes").data_ptr()) if g("nv_codes") is not None else None,
            P(g("nv_sf").data_ptr()) if g("nv_sf") is not None else None,
            P(g("nv_scale").data_ptr()) if g("nv_scale") is not None else None,
            P(g("mx_codes").data_ptr()) if g("mx_codes") is not None else None,
            P(g("mx_sf").data_ptr()) if g("mx_sf") is not None else None,
            seed, (bsq.SF_SWIZZLED if swz else 0) | (bsq.STOCHASTIC if sr else 0), None,
            P(torch.cuda.current_stream().cuda_stream))
    assert st == 0, st


@pytest.mark.gpu
def test_noalloc_matches_workspace_version_on_consecutive_calls(gpu, O):
    """Two calls in a row (the second with far smaller values, so column
    maxima left in the shared array by the first would change its FP32
    scales), then an MXFP8-only call, which leaves the array unused: each
    output equals requant_transpose_sr's, bit for bit, and the first call's
    equals the oracle's too.  Every output sits inside a guard band that must
    come back untouched."""
    bsq, fn = _fn()
    cases = [(256, 2048, 1.0, True, True, 7, True), (160, 768, 1e-3, True, False, 11, True),
             (128, 512, 1.0, False, True, 5, False)]
    for n, (rows, K, amp, sr, swz, seed, nv) in enumerate(cases):
        x = synth.to_bf16_bits(synth.bf16_bits_to_f32(synth.normal_with_outliers(rows, K, seed=seed)) * np.float32(amp))
        codes, sf, t = bsq.quantize_nvfp4_per_token(to_dev(x), swizzled=swz)
        ref = bsq.requant_transpose_sr(codes, sf, t, nvfp4=nv, stochastic=sr, seed=seed, swizzled=swz)
        guards = []
        out = {}
        for k, v in ref.items():
            if v is None:
                continue
            buf, view = guarded_empty(v.shape, v.dtype)
            guards.append(buf)
            out[k] = view
        _call(bsq, fn, codes, sf, t, rows, K, out, seed, sr, swz)
        torch.cuda.synchronize()
        for buf in guards:
            buf.check()
        for k, v in ref.items():
            if v is None:
                assert k not in out
                continue
            a, b = to_np(out[k]), to_np(v)
            assert bits_equal(a, b), f"{k} (rows={rows}, K={K}): {first_mismatch(a, b)}"
        if n == 0:
            oc, osf, ot = O.nvfp4_quantize_rows(x)
            nc, ns, nt, mc, ms = O.requant_transpose(oc, osf, ot, sr=sr, seed=seed)
            assert bits_equal(to_np(out["nv_codes"]), nc), "nv_codes vs oracle"
            assert bits_equal(to_np(out["nv_scale"]), nt), "nv_scale vs oracle"
            assert bits_equal(to_np(out["nv_sf"]), O.sf_to_swizzled(ns)), "nv_sf vs oracle"
            assert bits_equal(to_np(out["mx_codes"]), mc), "mx_codes vs oracle"
            assert bits_equal(to_np(out["mx_sf"]), O.sf_to_swizzled(ms)), "mx_sf vs oracle"
