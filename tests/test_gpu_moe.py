"""GPU: moe_expert_forward against the oracle, stage by stage.

A last-bit binary32 difference in the SwiGLU output h can legitimately flip
an NVFP4 code of h, so the forward is checked in stages: routing (exact),
quantize-scatter of x (bit-exact), GEMM1 + SwiGLU (GEMM tolerance + bf16),
quantization of the GPU's own h (bit-exact), GEMM2 from the GPU's own
quantized h (GEMM tolerance + bf16), combine of the GPU's own expert outputs
(fp32 accumulation + bf16 rounding).  With BSQ_MOE_FUSED_H GEMM1 quantizes h
in its epilogue instead; separate tests show that this changes no result bit
(with and without keeping h), and check those stages on the full-size
layers."""
import numpy as np
import pytest
import torch

from block_scaled_precision_quantize_gb300 import synth
from conftest import bits_equal, first_mismatch, to_dev, to_np

pytestmark = pytest.mark.gpu


def _ws(ws, L, field, dtype, shape):
    off = getattr(L, field)
    n = int(np.prod(shape)) * np.dtype(dtype).itemsize
    return to_np(ws[off:off + n]).view(dtype).reshape(shape)


def _unswz(O, sf_swz, rows, cols):
    """Inverse of the oracle's swizzle, via its offset function."""
    out = np.empty((rows, cols), np.uint8)
    r = np.arange(rows)[:, None]
    c = np.arange(cols)[None, :]
    ctiles = (cols + 3) // 4
    off = ((r // 128) * ctiles + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4
    out[:, :] = sf_swz[off]
    # the offset formula above must agree with the oracle's layout function
    assert O.sf_swizzled_offset(rows - 1, cols - 1, 16 * cols) == off[-1, -1]
    return out


def _bf16_bound(ref, ab, extra_rel=2.0 ** -8):
    return 1e-4 * ab + extra_rel * np.abs(ref) + 1e-30


class _ExpertQuant:
    """Oracle quantization of one expert's weights at a time (cached), checked
    bit-exact against the GPU per-expert quantizer's output for that expert."""

    def __init__(self, O, w_bits, gpu_q):
        self.O, self.w, self.g, self.cache, self.sf = O, w_bits, gpu_q, {}, None

    def __getitem__(self, e):
        if e not in self.cache:
            c, s, t = self.O.nvfp4_quantize_group(self.w[e:e + 1])
            N = self.w.shape[1]
            assert bits_equal(to_np(self.g[0][e]), c[0]) and bits_equal(to_np(self.g[2][e:e + 1]), t)
            if self.sf is None:
                self.sf = _unswz(self.O, to_np(self.g[1]), self.w.shape[0] * N, self.w.shape[2] // 16)
            assert bits_equal(self.sf[e * N:(e + 1) * N], s[0])
            self.cache[e] = (c[0], s[0], t[0])
        return self.cache[e]


def _staged(gpu, O, T, H, I, E, k, four_six, seed, sample_rows=None):
    x = synth.normal((T, H), seed=seed)
    ids, wts = synth.topk_routing(T, E, k, seed=seed)
    wgu_b = synth.normal((E, 2 * I, H), seed=seed + 1, std=0.02)
    wd_b = synth.normal((E, H, I), seed=seed + 2, std=0.02)
    wgu = gpu.quantize_nvfp4_per_expert(to_dev(wgu_b))
    wd = gpu.quantize_nvfp4_per_expert(to_dev(wd_b))
    # weights: oracle quantization per expert, bit-exact with the GPU's
    GU = _ExpertQuant(O, wgu_b, wgu)
    DN = _ExpertQuant(O, wd_b, wd)

    L = gpu.moe_workspace_layout(T, H, I, E, k)
    ws = torch.zeros(L.total, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = gpu.moe_expert_forward(to_dev(x), to_dev(ids), to_dev(wts), wgu, wd, I, four_six=four_six,
                               workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    cap = L.capacity

    # 1. routing
    offsets, slot_of, row_src = O.route(ids, E)
    R = int(offsets[-1])
    assert bits_equal(_ws(ws, L, "offsets", np.int32, (E + 1,)), offsets)
    assert bits_equal(_ws(ws, L, "slot_of", np.int32, (T * k,)), slot_of)
    assert bits_equal(_ws(ws, L, "row_src", np.int32, (cap,))[:R], row_src)

    # 2. quantize-scatter of x (per-token scales, 4/6 as requested)
    xc, xs, xt = O.nvfp4_quantize_rows(x, four_six=four_six)
    src_tok = np.where(row_src >= 0, row_src // k, -1)
    valid = src_tok >= 0
    q_codes = _ws(ws, L, "xq_codes", np.uint8, (cap, H // 2))[:R]
    q_scale = _ws(ws, L, "xq_scale", np.float32, (cap,))[:R]
    q_sf = _unswz(O, _ws(ws, L, "xq_sf", np.uint8, (cap * (H // 16),)), cap, H // 16)[:R]
    assert bits_equal(q_codes[valid], xc[src_tok[valid]]), first_mismatch(q_codes[valid], xc[src_tok[valid]])
    assert bits_equal(q_sf[valid], xs[src_tok[valid]])
    assert bits_equal(q_scale[valid], xt[src_tok[valid]])
    assert not q_sf[~valid].any() and not q_scale[~valid].any()

    rows = np.arange(R) if sample_rows is None else sample_rows(offsets, row_src)
    expert_of = np.searchsorted(offsets, rows, side="right") - 1

    # 3. GEMM1 + SwiGLU (on the oracle's own quantized x)
    h_gpu = _ws(ws, L, "h", np.uint16, (cap, I))
    ab = np.zeros((rows.size, 2 * I))
    ref = np.zeros((rows.size, 2 * I))
    for e in np.unique(expert_of):
        sel = np.where(expert_of == e)[0]
        rr = rows[sel]
        tok = np.maximum(src_tok[rr], 0)
        a_t = np.where(src_tok[rr] >= 0, xt[tok], 0).astype(np.float32)
        o, a = O.gemm_nvfp4(xc[tok], xs[tok], a_t, *GU[e])
        ref[sel], ab[sel] = o, a
    h_ref = O.swiglu(ref)
    g, u = ref[:, :I], ref[:, I:]
    sg = g / (1 + np.exp(-g))
    bound = 1.1 * np.abs(u) * 1e-4 * ab[:, :I] + np.abs(sg) * 1e-4 * ab[:, I:] + 2.0 ** -8 * np.abs(h_ref) + 1e-30
    hg = synth.bf16_bits_to_f32(h_gpu[rows]).astype(np.float64)
    assert np.all(np.abs(hg - h_ref) <= bound), np.max(np.abs(hg - h_ref) / bound)

    # 4. quantization of the GPU's own h (bit-exact)
    hc, hs, ht = O.nvfp4_quantize_rows(h_gpu[rows], four_six=four_six)
    hq_codes = _ws(ws, L, "hq_codes", np.uint8, (cap, I // 2))
    hq_scale = _ws(ws, L, "hq_scale", np.float32, (cap,))
    hq_sf = _unswz(O, _ws(ws, L, "hq_sf", np.uint8, (cap * (I // 16),)), cap, I // 16)
    assert bits_equal(hq_codes[rows], hc), first_mismatch(hq_codes[rows], hc)
    assert bits_equal(hq_sf[rows], hs) and bits_equal(hq_scale[rows], ht)

    # 5. GEMM2 from the GPU's own quantized h (bf16 expert outputs)
    out_gpu = _ws(ws, L, "out", np.uint16, (cap, H))
    for e in np.unique(expert_of):
        sel = np.where(expert_of == e)[0]
        rr = rows[sel]
        o, a = O.gemm_nvfp4(hq_codes[rr], hq_sf[rr], hq_scale[rr], *DN[e])
        got = synth.bf16_bits_to_f32(out_gpu[rr]).astype(np.float64)
        assert np.all(np.abs(got - o) <= _bf16_bound(o, a)), e

    # 6. combine of the GPU's own expert outputs
    if sample_rows is None:
        y_ref = O.combine(out_gpu, slot_of, wts)
        yg = synth.bf16_bits_to_f32(to_np(y)).astype(np.float64)
        yr = synth.bf16_bits_to_f32(y_ref).astype(np.float64)
        of = synth.bf16_bits_to_f32(out_gpu).astype(np.float64)
        terms = np.abs(of[slot_of.reshape(T, k)] * wts[:, :, None]).sum(axis=1)
        # both sides round to bf16 independently (GPU from its fp32 sum, the
        # oracle from fp64), so they may differ by one bf16 ulp <= 2^-7 |y|
        assert np.all(np.abs(yg - yr) <= 2.0 ** -7 * np.abs(yr) + 1e-6 * terms + 1e-30)
    return y


@pytest.mark.parametrize("four_six", [False, True])
def test_moe_staged_small(gpu, O, four_six):
    _staged(gpu, O, T=200, H=256, I=128, E=5, k=3, four_six=four_six, seed=11)


def test_moe_staged_skewed_routing(gpu, O):
    _staged(gpu, O, T=300, H=512, I=256, E=9, k=8, four_six=False, seed=4)


def test_moe_bad_expert_id_reported(gpu):
    T, H, I, E, k = 64, 256, 128, 4, 2
    x = synth.normal((T, H), seed=1)
    ids, wts = synth.topk_routing(T, E, k, seed=1)
    ids[5, 1] = 17
    wgu = gpu.quantize_nvfp4_per_expert(to_dev(synth.normal((E, 2 * I, H), seed=2, std=0.02)))
    wd = gpu.quantize_nvfp4_per_expert(to_dev(synth.normal((E, H, I), seed=3, std=0.02)))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = gpu.moe_expert_forward(to_dev(x), to_dev(ids), to_dev(wts), wgu, wd, I, dev_status=status)
    # bsq_check_status reads the word after the stream's work, and leaves it
    assert gpu.check_status(status) == gpu.DEV_BAD_EXPERT
    torch.cuda.synchronize()
    assert int(status.item()) == gpu.DEV_BAD_EXPERT
    assert torch.isfinite(y.float()).all()
    ids[5, 1] = 2
    status.zero_()
    gpu.moe_expert_forward(to_dev(x), to_dev(ids), to_dev(wts), wgu, wd, I, dev_status=status)
    assert gpu.check_status(status) == gpu.DEV_OK


def test_moe_qwen3_shaped_sampled(gpu, O):
    """The Qwen3-30B-A3B-shaped layer at full size (T=16384, H=2048, E=128,
    top-8, I=768), checked stage by stage on sampled routed rows: the most
    and least loaded experts and random rows."""
    def sample(offsets, row_src):
        g = np.random.default_rng(0)
        counts = np.diff(offsets)
        big, small = int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 1 << 30)))
        picks = [np.arange(offsets[big], offsets[big] + 48), np.arange(offsets[small], offsets[small] + 16),
                 g.choice(int(offsets[-1]), 192, replace=False)]
        return np.unique(np.concatenate(picks))
    _staged(gpu, O, T=16384, H=2048, I=768, E=128, k=8, four_six=False, seed=3, sample_rows=sample)


def test_moe_deepseek_shaped_sampled(gpu, O):
    """The DeepSeek-V3-shaped layer at full size (T=32768, H=7168, E=256,
    top-8 with a Zipf-skewed expert bias s=1.1, I=2048, 4/6 on the
    activations), weights drawn on the device.  Routing is checked in full;
    the later stages on sampled rows of four experts (the most and the least
    loaded and two random ones), whose weights alone go through the oracle.
    Per-token quantization is row-independent, so the oracle quantizes only
    the tokens those rows come from."""
    T, H, I, E, k, seed = 32768, 7168, 2048, 256, 8, 5
    x = synth.normal((T, H), seed=seed)
    ids, wts = synth.topk_routing(T, E, k, seed=seed, zipf_s=1.1)
    wgu_d = synth.device_normal_bf16((E, 2 * I, H), seed=51, std=0.02)
    wd_d = synth.device_normal_bf16((E, H, I), seed=52, std=0.02)
    wgu = gpu.quantize_nvfp4_per_expert(wgu_d)
    wd = gpu.quantize_nvfp4_per_expert(wd_d)
    L = gpu.moe_workspace_layout(T, H, I, E, k)
    ws = torch.zeros(L.total, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = gpu.moe_expert_forward(to_dev(x), to_dev(ids), to_dev(wts), wgu, wd, I, four_six=True, workspace=ws,
                               dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    cap = L.capacity

    # 1. routing (all pairs)
    offsets, slot_of, row_src = O.route(ids, E)
    R = int(offsets[-1])
    assert bits_equal(_ws(ws, L, "offsets", np.int32, (E + 1,)), offsets)
    assert bits_equal(_ws(ws, L, "slot_of", np.int32, (T * k,)), slot_of)
    assert bits_equal(_ws(ws, L, "row_src", np.int32, (cap,))[:R], row_src)

    # sampled rows: 32 from each of four experts (a segment holds its routed
    # rows first, then the padding up to a multiple of 128)
    counts = np.bincount(ids.ravel(), minlength=E)
    g = np.random.default_rng(1)
    big, small = int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 1 << 30)))
    others = [e for e in g.permutation(E) if counts[e] >= 32 and e not in (big, small)][:2]
    experts = [big, small] + [int(e) for e in others]
    rows = np.concatenate([offsets[e] + g.choice(int(counts[e]), min(32, int(counts[e])), replace=False)
                           for e in experts])
    src_tok = row_src[rows] // k
    assert np.all(row_src[rows] >= 0)

    # the sampled experts' weights, quantized by the oracle and checked bit-exact
    # against the GPU per-expert quantizer
    def expert_q(w_d, q, e):
        wb = to_np(w_d[e:e + 1].contiguous().view(torch.int16)).view(np.uint16)
        c, s, t = O.nvfp4_quantize_group(wb)
        N, Kc = w_d.shape[1], w_d.shape[2]
        assert bits_equal(to_np(q[0][e]), c[0]) and bits_equal(to_np(q[2][e:e + 1]), t)
        sf_all = to_np(q[1])
        nct = (Kc // 16 + 3) // 4
        tile_bytes = nct * 512
        r0 = e * N  # expert e's rows start on a 128-row tile boundary (N % 128 == 0)
        sf_e = _unswz(O, sf_all[(r0 // 128) * tile_bytes:((r0 + N) // 128) * tile_bytes], N, Kc // 16)
        assert bits_equal(sf_e, s[0])
        return c[0], s[0], t[0]

    # 2. quantize-scatter of the sampled rows' tokens, with 4/6
    xc, xs, xt = O.nvfp4_quantize_rows(x[src_tok], four_six=True)
    q_codes = _ws(ws, L, "xq_codes", np.uint8, (cap, H // 2))[rows]
    q_scale = _ws(ws, L, "xq_scale", np.float32, (cap,))[rows]
    q_sf = _unswz(O, _ws(ws, L, "xq_sf", np.uint8, (cap * (H // 16),)), cap, H // 16)[rows]
    assert bits_equal(q_codes, xc), first_mismatch(q_codes, xc)
    assert bits_equal(q_sf, xs) and bits_equal(q_scale, xt)

    h_gpu = _ws(ws, L, "h", np.uint16, (cap, I))
    hq_codes = _ws(ws, L, "hq_codes", np.uint8, (cap, I // 2))
    hq_scale = _ws(ws, L, "hq_scale", np.float32, (cap,))
    hq_sf = _unswz(O, _ws(ws, L, "hq_sf", np.uint8, (cap * (I // 16),)), cap, I // 16)
    out_gpu = _ws(ws, L, "out", np.uint16, (cap, H))
    base = 0
    for e in experts:
        n = min(32, int(counts[e]))
        sel = slice(base, base + n)
        rr = rows[sel]
        base += n
        GUe = expert_q(wgu_d, wgu, e)
        # 3. GEMM1 + SwiGLU on the oracle's own quantized x
        o, a = O.gemm_nvfp4(xc[sel], xs[sel], xt[sel], *GUe)
        h_ref = O.swiglu(o)
        gg, uu = o[:, :I], o[:, I:]
        sg = gg / (1 + np.exp(-gg))
        bound = 1.1 * np.abs(uu) * 1e-4 * a[:, :I] + np.abs(sg) * 1e-4 * a[:, I:] + 2.0 ** -8 * np.abs(h_ref) + 1e-30
        hg = synth.bf16_bits_to_f32(h_gpu[rr]).astype(np.float64)
        assert np.all(np.abs(hg - h_ref) <= bound), (e, np.max(np.abs(hg - h_ref) / bound))
        # 4. quantization of the GPU's own h, with 4/6 (bit-exact)
        hc, hs, ht = O.nvfp4_quantize_rows(h_gpu[rr], four_six=True)
        assert bits_equal(hq_codes[rr], hc) and bits_equal(hq_sf[rr], hs) and bits_equal(hq_scale[rr], ht), e
        # 5. GEMM2 from the GPU's own quantized h
        DNe = expert_q(wd_d, wd, e)
        o2, a2 = O.gemm_nvfp4(hq_codes[rr], hq_sf[rr], hq_scale[rr], *DNe)
        got = synth.bf16_bits_to_f32(out_gpu[rr]).astype(np.float64)
        assert np.all(np.abs(got - o2) <= _bf16_bound(o2, a2)), e

    # 6. combine of the GPU's own expert outputs, for the sampled rows' tokens
    toks = np.unique(src_tok)
    s_t = slot_of.reshape(T, k)[toks]
    w_t = wts[toks]
    y_ref = O.combine(out_gpu, s_t.reshape(-1), w_t)
    yg = synth.bf16_bits_to_f32(to_np(y)[toks]).astype(np.float64)
    yr = synth.bf16_bits_to_f32(y_ref).astype(np.float64)
    of = synth.bf16_bits_to_f32(out_gpu[s_t]).astype(np.float64)  # [tokens, k, H]: the sampled tokens only
    terms = np.abs(of * w_t[:, :, None]).sum(axis=1)
    assert np.all(np.abs(yg - yr) <= 2.0 ** -7 * np.abs(yr) + 1e-6 * terms + 1e-30)


def test_moe_staged_many_experts(gpu, O):
    """600 experts: the routing's single-warp slot assignment (beyond the
    CTA version's expert limit) and the GEMM's offsets read from global
    memory."""
    _staged(gpu, O, T=160, H=256, I=128, E=600, k=3, four_six=False, seed=8)


@pytest.mark.parametrize("four_six", [False, True])
def test_moe_fused_h_quantization_bit_identical(gpu, four_six):
    """BSQ_MOE_FUSED_H: GEMM1 quantizes h from its per-CTA scratch rows (or
    from the kept whole h with BSQ_MOE_KEEP_H).  The quantized h, the
    per-slot outputs and y equal, bit for bit, those of the two-pass path
    (GEMM1 -> bf16 h -> the per-token quantizer), which the staged tests
    check against the oracle (ragged experts, two N tiles per unit)."""
    T, H, I, E, k = 300, 512, 256, 9, 4
    x = synth.normal((T, H), seed=21)
    ids, wts = synth.topk_routing(T, E, k, seed=21)
    wgu = gpu.quantize_nvfp4_per_expert(to_dev(synth.normal((E, 2 * I, H), seed=22, std=0.02)))
    wd = gpu.quantize_nvfp4_per_expert(to_dev(synth.normal((E, H, I), seed=23, std=0.02)))
    L = gpu.moe_workspace_layout(T, H, I, E, k)
    outs = []
    for fused, keep in ((False, False), (True, False), (True, True)):
        ws = torch.zeros(L.total, dtype=torch.uint8, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        y = gpu.moe_expert_forward(to_dev(x), to_dev(ids), to_dev(wts), wgu, wd, I, four_six=four_six,
                                   workspace=ws, dev_status=status, fused_h=fused, keep_h=keep)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        R = int(_ws(ws, L, "offsets", np.int32, (E + 1,))[-1])
        outs.append((to_np(y), _ws(ws, L, "hq_codes", np.uint8, (L.capacity, I // 2))[:R],
                     _ws(ws, L, "hq_scale", np.float32, (L.capacity,))[:R],
                     _ws(ws, L, "hq_sf", np.uint8, (L.capacity * (I // 16),))[:R * (I // 16)],
                     _ws(ws, L, "out", np.uint16, (L.capacity, H))[:R]))
        if fused and not keep:
            assert not _ws(ws, L, "h", np.uint16, (L.capacity, I)).any()  # h itself never leaves the scratch
    for other in outs[1:]:
        for a, b, what in zip(outs[0], other, ("y", "hq codes", "hq scale", "hq sf", "per-slot outputs")):
            assert bits_equal(a, b), what


def test_moe_fused_h_quantization_bit_identical_full_size(gpu):
    """The same identity on the Qwen3-30B-A3B-shaped layer (T=16384, H=2048,
    E=128, top-8, I=768): 576 pair units of six N tiles each."""
    T, H, I, E, k = 16384, 2048, 768, 128, 8
    x = synth.normal((T, H), seed=3)
    ids, wts = synth.topk_routing(T, E, k, seed=3)
    wgu = gpu.quantize_nvfp4_per_expert(synth.device_normal_bf16((E, 2 * I, H), seed=31, std=0.02))
    wd = gpu.quantize_nvfp4_per_expert(synth.device_normal_bf16((E, H, I), seed=32, std=0.02))
    L = gpu.moe_workspace_layout(T, H, I, E, k)
    res = []
    for fused in (False, True):
        ws = torch.zeros(L.total, dtype=torch.uint8, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        y = gpu.moe_expert_forward(to_dev(x), to_dev(ids), to_dev(wts), wgu, wd, I, workspace=ws, dev_status=status,
                                   fused_h=fused)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        R = int(_ws(ws, L, "offsets", np.int32, (E + 1,))[-1])
        res.append((y.clone(), ws[L.hq_codes:L.hq_codes + R * (I // 2)].clone(),
                    ws[L.hq_scale:L.hq_scale + 4 * R].clone(), ws[L.hq_sf:L.hq_sf + R * (I // 16)].clone()))
        del ws
    for a, b, what in zip(res[0], res[1], ("y", "hq codes", "hq scale", "hq sf")):
        assert torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                           b.view(torch.uint8) if b.dtype != torch.uint8 else b), what


@pytest.mark.parametrize("fused", [False, True])
def test_moe_workspace_guard_bands(gpu, fused):
    """Every sub-buffer of the MoE workspace is followed by unused bytes: the
    forward, run on a workspace filled with a canary byte, must leave all of
    them, from the end of each sub-buffer's data to the next sub-buffer, as
    they were (the writes stay inside their buffers, in both GEMM1 paths)."""
    from conftest import CANARY
    T, H, I, E, k = 200, 256, 128, 5, 3
    x = synth.normal((T, H), seed=11)
    ids, wts = synth.topk_routing(T, E, k, seed=11)
    wgu = gpu.quantize_nvfp4_per_expert(to_dev(synth.normal((E, 2 * I, H), seed=12, std=0.02)))
    wd = gpu.quantize_nvfp4_per_expert(to_dev(synth.normal((E, H, I), seed=13, std=0.02)))
    L = gpu.moe_workspace_layout(T, H, I, E, k)
    cap = L.capacity
    ceil4 = lambda n: (n + 3) // 4 * 4  # noqa: E731
    nchunks = max((T * k + 511) // 512, 1)
    sizes = {"offsets": (E + 1) * 4, "counts": E * 4, "slot_of": T * k * 4, "row_src": cap * 4,
             "xq_codes": cap * H // 2, "xq_sf": cap * ceil4(H // 16), "xq_scale": cap * 4, "h": cap * I * 2,
             "hq_codes": cap * I // 2, "hq_sf": cap * ceil4(I // 16), "hq_scale": cap * 4, "out": cap * H * 2,
             "scan": (nchunks * E + 1) * 4, "h_scratch": 2 * 256 * 128 * I * 2}
    fields = sorted(sizes, key=lambda f: getattr(L, f))
    ws = torch.full((L.total,), CANARY, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu.moe_expert_forward(to_dev(x), to_dev(ids), to_dev(wts), wgu, wd, I, workspace=ws, dev_status=status,
                           fused_h=fused)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    w = to_np(ws)
    for f, nxt in zip(fields, fields[1:] + [None]):
        end = getattr(L, f) + sizes[f]
        stop = getattr(L, nxt) if nxt else L.total
        assert stop - end >= 256, f
        gap = w[end:stop]
        assert np.all(gap == CANARY), f"write past the end of workspace buffer {f}: {int((gap != CANARY).sum())} bytes"
