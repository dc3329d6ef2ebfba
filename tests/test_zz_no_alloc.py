"""requant_transpose_sr_noalloc: the allocation-free entry point for callers
that cannot give the library device scratch memory (a host framework that
owns only its input and output buffers, or code that must not allocate
device memory once running).  It keeps the column maxima in a fixed array
inside the library, so it takes no workspace; its results must equal those of
requant_transpose_sr.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from block_scaled_precision_quantize_gb300 import synth
from conftest import bits_equal, first_mismatch, to_dev, to_np

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


def test_noalloc_rejects_k_beyond_its_array():
    _, fn = _fn()
    d = P(4096)
    assert fn(d, d, d, 64, 65536 + 16, d, d, d, None, None, 0, 0, None, None) == 2  # BSQ_ERR_SHAPE
    assert fn(d, d, d, 64, 96, d, d, d, None, None, 0, 1 << 9, None, None) == 4     # BSQ_ERR_FLAGS


@pytest.mark.gpu
def test_noalloc_matches_workspace_version_on_consecutive_calls(gpu):
    bsq, fn = _fn()
    stream = P(torch.cuda.current_stream().cuda_stream)
    # the second call has much smaller values: stale column maxima left in
    # the shared array by the first call would change its FP32 scales
    cases = [(256, 2048, 1.0, True, True, 7), (160, 768, 1e-3, True, False, 11)]
    for rows, K, amp, sr, swz, seed in cases:
        x = synth.to_bf16_bits(synth.bf16_bits_to_f32(synth.normal_with_outliers(rows, K, seed=seed)) * np.float32(amp))
        codes, sf, t = bsq.quantize_nvfp4_per_token(to_dev(x), swizzled=swz)
        ref = bsq.requant_transpose_sr(codes, sf, t, stochastic=sr, seed=seed, swizzled=swz)
        out = {k: torch.empty_like(v) for k, v in ref.items()}
        st = fn(P(codes.data_ptr()), P(sf.data_ptr()), P(t.data_ptr()), rows, K, P(out["nv_codes"].data_ptr()),
                P(out["nv_sf"].data_ptr()), P(out["nv_scale"].data_ptr()), P(out["mx_codes"].data_ptr()),
                P(out["mx_sf"].data_ptr()), seed, (bsq.SF_SWIZZLED if swz else 0) | (bsq.STOCHASTIC if sr else 0),
                None, stream)
        assert st == 0, st
        torch.cuda.synchronize()
        for k in ("nv_codes", "nv_sf", "nv_scale", "mx_codes", "mx_sf"):
            a, b = to_np(out[k]), to_np(ref[k])
            assert bits_equal(a, b), f"{k} (rows={rows}, K={K}): {first_mismatch(a, b)}"
