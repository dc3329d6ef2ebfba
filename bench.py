#!/usr/bin/env python3
"""Benchmark of the block-scaled MoE expert hot path on GB300; prints ONE JSON
line on rank 0.

A step is one moe_expert_forward over the Qwen3-30B-A3B-shaped expert layer
(T=16384 tokens, H=2048, E=128 experts, top-8, I=768): routing, per-token
NVFP4 quantization of x into the routed slots, the tcgen05 grouped GEMM with
gate/up weights and the fused SwiGLU + FP32 rescale, per-token NVFP4 of h, the
grouped GEMM with down weights, and the weighted combine.  value = the two
GEMMs' algorithmic FLOPs / step time (TFLOP/s), summed over all ranks (each
rank runs its own replica: weak scaling, no collective on the data path).
The working set (~0.9 GB: weights, activations, workspace) is larger than the
129 MB L2, so no flush is needed between steps.

Also reported: per-stage times (CUDA events the library records at the
stage boundaries on the launching stream, from a second pass right after the
timed one), each data-moving stage's HBM floor (its bytes at the measured copy
rate, or its written bytes at the write-only rate measured in the same run,
whichever takes longer), a roofline for the dominant kernel, the standalone quantizers (MXFP8 row+col on 16384x2048, NVFP4
per-token on 16384x2048, requant with Philox SR and round-to-nearest on
16384x2048 and 16384x768; back-to-back launches through the C ABI rotating
over input/output sets larger than twice the L2, so every launch starts
cold), an end-to-end number through the public API
with pinned-host inputs/outputs copied inside the timed region, SM clocks
sampled during the timed region, and the CPU oracle's throughput on a
bounded sample.

--impl reference times the CPU oracle instead (on the host cores, rank 0
only) on a bounded per-step sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "NVFP4 grouped expert GEMM TFLOPS + quantize GB/s, % of GB300 roofline"
WORKLOADS = {
    "qwen3": dict(T=16384, H=2048, E=128, k=8, I=768, seed=3, w_seed_gu=31, w_seed_d=32,
                  name="Qwen3-30B-A3B-shaped MoE expert layer (T=16384, H=2048, E=128, top-8, I=768)"),
    "deepseek": dict(T=32768, H=7168, E=256, k=8, I=2048, seed=5, w_seed_gu=51, w_seed_d=52, zipf=1.1,
                     four_six=True,
                     name="DeepSeek-V3-shaped MoE expert layer (T=32768, H=7168, E=256, top-8, I=2048, 4/6)"),
}
KERNELS_PER_STEP = 8  # route x3, quantize-scatter (with the padding rows), GEMM1, quantize h, GEMM2, combine


def gemm_flops(w):
    R = w["T"] * w["k"]
    return 2.0 * R * (2 * w["I"]) * w["H"], 2.0 * R * w["H"] * w["I"]


def peaks():
    """HBM and tensor peaks.  The tensor-bound kernels are timed in short
    bursts (the whole timed region is milliseconds), so their denominators
    are burst figures: the block-scaled MMA ceiling measured in this run
    (measure_mma_ceiling) replaces these until it is available; the
    fallback is the burst bf16 peak x the nominal FP4/BF16 (6) or FP8/BF16
    (2) ratio."""
    p = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        p.update({k: m[k] for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained") if k in m})
        p["source"] = "measured"
    p["fp4_tflops"] = p["bf16_tflops"] * 6.0
    p["fp4_source"] = f"{p['source']} bf16 burst x 6 (nominal FP4/BF16 ratio)"
    p["fp8_tflops"] = p["bf16_tflops"] * 2.0
    p["fp8_source"] = f"{p['source']} bf16 burst x 2 (nominal FP8/BF16 ratio)"
    return p


def measure_mma_ceiling(bsq, dev, P, iters=4096, reps=10):
    """The block-scaled MMA ceiling of this GPU (bsq_mma_ceiling): one CTA
    per SM issuing back-to-back MMAs of the GEMM's forms, timed with CUDA
    events on the launching stream; also the per-MMA cycles from the
    kernel's clock64 records.  Sets P's fp4/fp8 peaks to the best form of
    each format."""
    import torch
    flops_per_mma = {0: 2.0 * 128 * 256 * 64, 1: 2.0 * 128 * 256 * 32}
    out = {}
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for fmt, fname in ((0, "nvfp4"), (1, "mxfp8")):
        for cg in (1, 2):
            for _ in range(3):
                bsq.mma_ceiling(fmt, cg, iters, device=dev, dev_status=status)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * reps)]
            runs = []
            torch.cuda.synchronize()
            for r in range(reps):
                ev[2 * r].record()
                ctas, cyc = bsq.mma_ceiling(fmt, cg, iters, device=dev, dev_status=status)
                ev[2 * r + 1].record()
                runs.append(cyc)
            torch.cuda.synchronize()
            ms = min(ev[2 * r].elapsed_time(ev[2 * r + 1]) for r in range(reps))
            issuing = [int(c) for c in runs[-1].cpu().tolist() if int(c) > 0]
            tflops = ctas * iters * flops_per_mma[fmt] / (ms * 1e-3) / 1e12
            out[f"{fname}_cta_group_{cg}"] = {
                "tflops": tflops, "us_per_launch": ms * 1e3, "ctas": ctas, "mmas_per_cta": iters,
                "cycles_per_mma": statistics.median(issuing) / iters if issuing else None,
                "shape_per_cta": f"128x256x{64 if fmt == 0 else 32}"}
    assert int(status.item()) == 0, f"MMA ceiling: device status {int(status.item())}"
    best4 = max(out["nvfp4_cta_group_1"]["tflops"], out["nvfp4_cta_group_2"]["tflops"])
    best8 = max(out["mxfp8_cta_group_1"]["tflops"], out["mxfp8_cta_group_2"]["tflops"])
    P["fp4_tflops"], P["fp8_tflops"] = best4, best8
    P["fp4_source"] = "measured in this run: back-to-back tcgen05.mma kind::mxf4nvf4 (bsq_mma_ceiling), best form"
    P["fp8_source"] = "measured in this run: back-to-back tcgen05.mma kind::mxf8f6f4 (bsq_mma_ceiling), best form"
    return out


def measure_write_bw(dev, P, nbytes=1 << 31, reps=5):
    """HBM write-only rate of this GPU: a fill of a 2 GiB buffer (torch's
    fill kernel, one value throughout; bytes written / CUDA-event time, best
    of `reps`).  Stored in P as the denominator of the write side of a
    stage's HBM floor; data that varies may write more slowly, so the floor
    it gives is a lower bound on the time."""
    import torch
    buf = torch.empty(nbytes // 4, dtype=torch.int32, device=dev)
    for _ in range(2):
        buf.fill_(1)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * reps)]
    torch.cuda.synchronize()
    for r in range(reps):
        ev[2 * r].record()
        buf.fill_(r)
        ev[2 * r + 1].record()
    torch.cuda.synchronize()
    ms = min(ev[2 * r].elapsed_time(ev[2 * r + 1]) for r in range(reps))
    del buf
    P["hbm_write_gbs"] = nbytes / (ms * 1e-3) / 1e9
    P["hbm_write_source"] = "measured in this run: fill of a 2 GiB buffer, bytes written / time, best of 5"
    return P["hbm_write_gbs"]


STAGES = ["route", "quantize_scatter", "gemm1_swiglu", "quantize_h", "gemm2", "combine"]


def stage_traffic(w, R_pad):
    """Algorithmic HBM bytes (read, written) of the forward's stages that
    move data: x read once and each routed copy of its codes, scale factors
    and token scale written; h read and quantized; GEMM2's A, weights and
    bf16 per-slot outputs; the per-slot outputs gathered and y written."""
    T, H, I, E, k = w["T"], w["H"], w["I"], w["E"], w["k"]
    R = T * k
    return {"quantize_scatter": (T * H * 2, R * (H // 2 + H // 16 + 4)),
            "quantize_h": (R_pad * I * 2, R_pad * (I // 2 + I // 16 + 4)),
            "gemm2": (R_pad * (I // 2 + I // 16 + 4) + E * H * (I // 2 + I // 16), R_pad * H * 2),
            "combine": (R * H * 2 + R * 8, T * H * 2)}


def stage_table(ev, w, R_pad, P):
    """Mean stage times over the event rows `ev`, with each stage's rate:
    TFLOP/s for the GEMMs; for the stages that move data, GB/s against the
    measured copy rate, and the HBM floor, the longer of (all bytes at the
    copy rate) and (the bytes written at the write-only rate)."""
    f1, f2 = gemm_flops(w)
    traffic = stage_traffic(w, R_pad)
    stages = {}
    for s, n in enumerate(STAGES):
        ms = statistics.mean(row[s].elapsed_time(row[s + 1]) for row in ev)
        d = {"ms": ms}
        if n in ("gemm1_swiglu", "gemm2"):
            d["tflops"] = (f1 if n == "gemm1_swiglu" else f2) / (ms * 1e-3) / 1e12
            d["frac_of_fp4_peak"] = d["tflops"] / P["fp4_tflops"]
        if n in traffic:
            rd, wr = traffic[n]
            if n != "gemm2":
                d["gbs"] = (rd + wr) / (ms * 1e-3) / 1e9
                d["frac_of_hbm"] = d["gbs"] / P["hbm_gbs"]
            if "hbm_write_gbs" in P:
                floor = max((rd + wr) / (P["hbm_gbs"] * 1e9), wr / (P["hbm_write_gbs"] * 1e9)) * 1e3
                d["hbm_floor_ms"] = floor
                d["frac_of_hbm_floor"] = floor / ms
        stages[n] = d
    return stages


# ----------------------------------------------------------------- clocks
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.idx)], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(self.NAMES, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- distributed
def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- CPU oracle
def oracle_expert_pass(O, x_bits, rows_tok, wgu_q, wd_q, four_six):
    """The oracle on one expert's routed rows: per-token NVFP4 of x, GEMM1
    (fp64 on exact dequantized operands), SwiGLU, bf16 h, per-token NVFP4
    of h, GEMM2.  Returns the FLOPs done."""
    xq = O.nvfp4_quantize_rows(x_bits[rows_tok], four_six=four_six)
    gu, _ = O.gemm_nvfp4(*xq, *wgu_q, with_abs=False)
    h = O.f64_to_bf16_array(O.swiglu(gu))
    hq = O.nvfp4_quantize_rows(h, four_six=four_six)
    O.gemm_nvfp4(*hq, *wd_q, with_abs=False)
    n, I2, H = rows_tok.size, wgu_q[0].shape[0], x_bits.shape[1]
    return 2.0 * n * I2 * H + 2.0 * n * H * (I2 // 2)


def oracle_setup(w, experts, x_bits=None, ids=None):
    """Inputs for the oracle legs: x and routing from the workload's seeds,
    the sampled experts' weights drawn on the host with the same
    distribution, quantized by the oracle (untimed)."""
    import oracle as O
    from block_scaled_precision_quantize_gb300 import synth
    O.build()
    T, H, I, E, k = w["T"], w["H"], w["I"], w["E"], w["k"]
    if x_bits is None:
        x_bits = synth.normal((T, H), seed=w["seed"])
    if ids is None:
        ids, _ = synth.topk_routing(T, E, k, seed=w["seed"], zipf_s=w.get("zipf"))
    qs = {}
    for e in experts:
        gu = synth.normal((1, 2 * I, H), seed=w["w_seed_gu"], stream=1000 + e, std=0.02)
        dn = synth.normal((1, H, I), seed=w["w_seed_d"], stream=1000 + e, std=0.02)
        c, s, t = O.nvfp4_quantize_group(gu)
        c2, s2, t2 = O.nvfp4_quantize_group(dn)
        qs[e] = ((c[0], s[0], t[0]), (c2[0], s2[0], t2[0]))
    tok_of = {e: np.nonzero((ids == e).any(axis=1))[0] for e in experts}
    return O, x_bits, qs, tok_of


def cpu_info():
    """Host core count and CPU model (lscpu's "Model name", else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None and os.path.exists("/proc/cpuinfo"):
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
    return {"nproc": os.cpu_count(), "cpu_model": model}


def _oracle_expert_job(job):
    """One expert's whole routed segment through the oracle, in a worker
    process (spawned: no CUDA state is inherited).  Returns its FLOPs."""
    w, e, x_rows = job
    import oracle as O
    from block_scaled_precision_quantize_gb300 import synth
    O.build()
    I, H = w["I"], w["H"]
    gu = synth.normal((1, 2 * I, H), seed=w["w_seed_gu"], stream=1000 + e, std=0.02)
    dn = synth.normal((1, H, I), seed=w["w_seed_d"], stream=1000 + e, std=0.02)
    c, s_, t = O.nvfp4_quantize_group(gu)
    c2, s2, t2 = O.nvfp4_quantize_group(dn)
    return oracle_expert_pass(O, x_rows, np.arange(x_rows.shape[0]), (c[0], s_[0], t[0]), (c2[0], s2[0], t2[0]),
                              w.get("four_six", False))


def oracle_all_cores(w, x_bits, ids, nproc):
    """The same oracle on every host core: one expert's routed segment per
    worker process, experts 0 .. nproc-1 at once; value = their FLOPs / the
    wall time of the parallel pass (pool start-up excluded)."""
    import multiprocessing as mp
    experts = list(range(min(w["E"], nproc)))
    jobs = [(w, e, x_bits[np.nonzero((ids == e).any(axis=1))[0]]) for e in experts]
    ctx = mp.get_context("spawn")
    with ctx.Pool(nproc) as pool:
        pool.map(abs, range(nproc))  # workers up before the clock starts
        t0 = time.perf_counter()
        flops = sum(pool.map(_oracle_expert_job, jobs, chunksize=1))
        dt = time.perf_counter() - t0
    rows = sum(j[2].shape[0] for j in jobs)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": nproc, "seconds": dt,
            "sample": f"experts 0..{experts[-1]}, one whole routed segment per process ({rows} rows), "
                      f"{flops / 1e9:.1f} GFLOP"}


def oracle_per_config(budget_each_s=4.0):
    """Single-core oracle times on bounded samples of each workload's
    quantization or GEMM work, in the units the GPU figures use."""
    import oracle as O
    from block_scaled_precision_quantize_gb300 import synth
    O.build()
    res = {}

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    # tiny single-expert path, whole: x 64x256 per-token, W 128x256 per-expert, GEMM 64x128
    x = synth.normal_with_outliers(64, 256, seed=0, stream=0)
    wt = synth.normal((1, 128, 256), seed=0, stream=1, std=0.02)

    def tiny():
        a = O.nvfp4_quantize_rows(x)
        b = O.nvfp4_quantize_group(wt)
        O.gemm_nvfp4(*a, b[0][0], b[1][0], b[2][0])
    res["tiny_64x256_gemm_64x128"] = {"ms": timed(tiny) * 1e3, "sample": "whole workload"}

    def rate(name, rows_total, K, make, run, bytes_per_row, note, cap=None):
        rows = 64
        xs = make(rows)
        dt = timed(lambda: run(xs))
        while dt < budget_each_s / 4 and rows * 2 <= min(rows_total, cap or rows_total):
            rows *= 2
            xs = make(rows)
            dt = timed(lambda: run(xs))
        res[name] = {"gbs": rows * bytes_per_row / dt / 1e9, "s": dt,
                     "sample": f"{rows} of {rows_total} rows x {K}; {note}"}

    x2 = synth.rows_log_uniform_std(16384, 2048, seed=2)
    rate("mxfp8_rowcol_16384x2048", 16384, 2048, lambda r: x2[:r], lambda a: O.mxfp8_quantize_rowcol(a),
         2048 * 4.0625, "row + column copies")
    x3 = synth.normal((16384, 2048), seed=3)
    rate("qwen3_x_nvfp4_16384x2048", 16384, 2048, lambda r: x3[:r], lambda a: O.nvfp4_quantize_rows(a),
         2048 * 2 + 1024 + 128 + 4, "per-token NVFP4 of the layer's x")
    x4 = synth.normal_with_outliers(16384, 2048, seed=7)
    q4 = O.nvfp4_quantize_rows(x4[:4096])
    rate("requant_sr_16384x2048", 16384, 2048, lambda r: (q4[0][:r], q4[1][:r], q4[2][:r]),
         lambda a: O.requant_transpose(*a, sr=True, seed=7),
         (1024 + 128 + 4) + (1024 + 128 + 4) + (2048 + 64), "dequantize, transpose, NVFP4 + MXFP8 with SR",
         cap=4096)
    x5 = synth.normal((2048, 7168), seed=5)
    rate("deepseek_x_nvfp4_4over6_32768x7168", 32768, 7168, lambda r: x5[:r],
         lambda a: O.nvfp4_quantize_rows(a, four_six=True), 7168 * 2 + 3584 + 448 + 4,
         "per-token NVFP4 with 4/6 of the layer's x", cap=2048)
    return res


def cpu_baseline(w, x_bits, ids, budget_s=12.0):
    """The oracle, as it stands, on whole routed segments of experts 0, 1, ...
    until about budget_s seconds of work on one host thread; then the same
    oracle on every core, and single-core figures for the other workloads."""
    experts = [0, 1, 2]
    O, x_bits, qs, tok_of = oracle_setup(w, experts, x_bits, ids)
    flops, t0, used = 0.0, time.perf_counter(), []
    for e in experts:
        flops += oracle_expert_pass(O, x_bits, tok_of[e], *qs[e], w.get("four_six", False))
        used.append(e)
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    rows = int(sum(tok_of[e].size for e in used))
    info = cpu_info()
    out = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
           "sample": f"experts {used} whole routed segments ({rows} rows) through NVFP4 quantize, GEMM1, "
                     f"SwiGLU, h quantize, GEMM2 on one host thread ({dt:.1f} s, {flops / 1e9:.1f} GFLOP)",
           **info}
    if info["nproc"] and info["nproc"] > 1:
        out["all_cores"] = oracle_all_cores(w, x_bits, ids, info["nproc"])
    out["per_config_single_core"] = oracle_per_config()
    return out


def run_reference(args, w, rank, world):
    """Reference arm: the oracle on the host cores, rank 0 only."""
    if rank != 0:
        return
    K, W = args.steps, args.warmup
    budget = 90.0
    rows_per_step = int(max(1, min(256, (budget / max(1, K + W) - 0.12) / 0.004)))
    experts = list(range(min(w["E"], 8)))
    O, x_bits, qs, tok_of = oracle_setup(w, experts)
    four_six = w.get("four_six", False)

    def step(i):
        e = experts[i % len(experts)]
        toks = tok_of[e][: rows_per_step]
        return oracle_expert_pass(O, x_bits, toks, *qs[e], four_six)

    for i in range(W):
        step(i)
    flops, t0 = 0.0, time.perf_counter()
    for i in range(K):
        flops += step(i)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = (f"per step: {rows_per_step} routed rows of one expert (rotating over experts {experts[0]}..{experts[-1]}) "
              f"through NVFP4 quantize, GEMM1, SwiGLU, h quantize, GEMM2, one host thread")
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "impl": "reference", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": dt / K * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w["name"], "T": w["T"], "H": w["H"], "E": w["E"], "topk": w["k"], "I": w["I"]},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "sample": sample,
                             **cpu_info()},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU arm
def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "block_scaled_precision_quantize_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_record(kernel_key, src_hash):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel_key)
    if not rec or rec.get("source_hash") != src_hash:
        return None
    return rec.get("dram_bytes_per_launch")


def run_ours(args, w, rank, world, local):
    import torch

    import block_scaled_precision_quantize_gb300 as bsq
    from block_scaled_precision_quantize_gb300 import synth

    bsq.build()
    bsq.load()
    dev = torch.device("cuda", local)
    T, H, I, E, k = w["T"], w["H"], w["I"], w["E"], w["k"]
    four_six = w.get("four_six", False)
    P = peaks()

    # inputs (synthetic, seeded): x and routing on the host, weights on the device
    x_bits = synth.normal((T, H), seed=w["seed"])
    ids, wts = synth.topk_routing(T, E, k, seed=w["seed"], zipf_s=w.get("zipf"))
    x_host = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    ids_host = torch.from_numpy(ids).pin_memory()
    wts_host = torch.from_numpy(wts).pin_memory()
    x = x_host.to(dev)
    ids_d = ids_host.to(dev)
    wts_d = wts_host.to(dev)
    wgu_b = synth.device_normal_bf16((E, 2 * I, H), seed=w["w_seed_gu"], std=0.02, device=dev)
    wgu = bsq.quantize_nvfp4_per_expert(wgu_b)
    del wgu_b
    wd_b = synth.device_normal_bf16((E, H, I), seed=w["w_seed_d"], std=0.02, device=dev)
    wd = bsq.quantize_nvfp4_per_expert(wd_b)
    del wd_b
    ws = torch.empty(bsq.moe_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=dev)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()

    def fwd(x=x, ids_d=ids_d, wts_d=wts_d, y=y):
        bsq.moe_expert_forward(x, ids_d, wts_d, wgu, wd, I, four_six=four_six, workspace=ws, y=y, dev_status=status)

    K, Wm = args.steps, args.warmup
    for _ in range(Wm):
        fwd()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    clocks = Clocks(f"GPU-{uuid}" if uuid is not None else local)
    clocks.start()
    # the step as a caller runs it, with no events between the forward's
    # kernels (recording events at the six stage boundaries added ~14 us to
    # a 0.66 ms step)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record()
    for i in range(K):
        fwd()
    t_end.record()
    torch.cuda.synchronize()
    barrier(world)
    ms_step = max_over_ranks(t_start.elapsed_time(t_end) / K, world)
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    # the per-stage breakdown (and the roofline's per-launch kernel time),
    # from a second pass right after the timed one, with events at the stage
    # boundaries on the forward's stream; the clock sampler covers both passes
    Ks = min(K, 20)
    stage_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(Ks)]
    for row in stage_ev:
        for e in row:
            e.record()
    torch.cuda.synchronize()
    for i in range(Ks):
        bsq.set_stage_events(stage_ev[i])
        fwd()
    bsq.set_stage_events(None)
    torch.cuda.synchronize()
    # the roofline's tensor denominators and the write-only HBM rate,
    # measured under the same clock sampling
    ceiling = measure_mma_ceiling(bsq, dev, P)
    measure_write_bw(dev, P)
    clk = clocks.stop()
    # the same step with h quantized inside GEMM1's epilogue (moe_expert_forward
    # with BSQ_MOE_FUSED_H: bit-identical results), timed for comparison
    fe0, fe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        bsq.moe_expert_forward(x, ids_d, wts_d, wgu, wd, I, four_six=four_six, workspace=ws, y=y, dev_status=status,
                               fused_h=True)
    fe0.record()
    for _ in range(Ks):
        bsq.moe_expert_forward(x, ids_d, wts_d, wgu, wd, I, four_six=four_six, workspace=ws, y=y, dev_status=status,
                               fused_h=True)
    fe1.record()
    torch.cuda.synchronize()
    fused_h_ms = fe0.elapsed_time(fe1) / Ks
    f1, f2 = gemm_flops(w)
    flops = f1 + f2
    value = flops * world / (ms_step * 1e-3) / 1e12

    R = T * k
    L = bsq.moe_workspace_layout(T, H, I, E, k)
    offsets = torch.empty(E + 1, dtype=torch.int32)
    offsets.copy_(ws[L.offsets:L.offsets + 4 * (E + 1)].view(torch.int32))
    R_pad = int(offsets[-1])
    stages = stage_table(stage_ev, w, R_pad, P)
    stage_ms = {n: d["ms"] for n, d in stages.items()}

    # roofline of the dominant kernel
    dom = max(STAGES, key=lambda n: stage_ms[n])
    gemm_hash = source_hash("gemm_fp4.cu", "common.cuh", "tc_ptx.cuh")
    if dom in ("gemm1_swiglu", "gemm2"):
        fl = f1 if dom == "gemm1_swiglu" else f2
        ach = fl / (stage_ms[dom] * 1e-3) / 1e12
        tr = traffic_record(f"k_gemm_fp4:{dom}:{args.workload}", gemm_hash)
        roof = {"kernel": f"k_gemm_fp4 ({dom})", "bound": "tensor", "achieved": ach,
                "peak": P["fp4_tflops"], "unit": "TFLOP/s", "frac": ach / P["fp4_tflops"],
                "traffic": tr, "peak_source": P["fp4_source"],
                "frac_of_bf16_burst_x6": ach / (P["bf16_tflops"] * 6.0),
                "frac_of_page_15pf": ach / 15000.0}
    else:
        ach = stages[dom].get("gbs", 0.0)
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": P["hbm_gbs"], "unit": "GB/s",
                "frac": ach / P["hbm_gbs"], "traffic": None, "peak_source": P["source"]}

    # End to end through the public API: every step's inputs are copied from
    # pinned host memory and its output back to pinned host memory, all inside
    # the timed region.  The copies run on their own streams into two buffer
    # sets, so step i+1's upload and step i-1's download overlap step i's
    # forward, as a serving pipeline runs them; events order each buffer's
    # reuse after the work that read it.
    main = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    xs, idss, wtss, ys = [x, torch.empty_like(x)], [ids_d, torch.empty_like(ids_d)], [wts_d, torch.empty_like(wts_d)], \
        [y, torch.empty_like(y)]
    y_host = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    Ke = max(3, min(K, 30))

    def e2e_steps(n):
        in_done = [torch.cuda.Event() for _ in range(n)]
        fwd_done = [torch.cuda.Event() for _ in range(n)]
        out_done = [torch.cuda.Event() for _ in range(n)]

        def upload(i):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(fwd_done[i - 2])  # the forward that read this buffer set is done
                xs[b].copy_(x_host, non_blocking=True)
                idss[b].copy_(ids_host, non_blocking=True)
                wtss[b].copy_(wts_host, non_blocking=True)
                in_done[i].record(s_in)

        s_in.wait_stream(main)  # nothing is copied before the timed region starts
        upload(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                upload(i + 1)
            main.wait_event(in_done[i])
            if i >= 2:
                main.wait_event(out_done[i - 2])  # this output buffer's previous download is done
            fwd(xs[b], idss[b], wtss[b], ys[b])
            fwd_done[i].record(main)
            with torch.cuda.stream(s_out):
                s_out.wait_event(fwd_done[i])
                y_host[b].copy_(ys[b], non_blocking=True)
                out_done[i].record(s_out)
        main.wait_event(out_done[n - 1])

    e2e_steps(2)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    e2e_steps(Ke)
    e1.record()
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / Ke, world)
    # every step saw the same inputs: the last download must equal the device forward's output
    if not torch.equal(y_host[(Ke - 1) % 2], ys[(Ke - 1) % 2].cpu()):
        raise RuntimeError("end-to-end output differs from the device forward's")
    e2e = {"value": flops * world / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms_e2e,
           "h2d_bytes_per_step": T * H * 2 + ids.nbytes + wts.nbytes, "d2h_bytes_per_step": T * H * 2,
           "copies": "double-buffered on two copy streams, overlapping the forwards"}

    components = {} if args.no_components else {**quantizer_components(bsq, synth, dev, P),
                                                 **backward_gemm_components(bsq, dev, P)}
    # the other layer shape the pages run (DeepSeek-V3-shaped, 4/6 on the
    # activations) as a second record, when this run is the Qwen3 one
    second = None
    if not args.no_components and args.workload == "qwen3" and world == 1:
        second = layer_record(bsq, synth, WORKLOADS["deepseek"], dev, P)

    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": Wm,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "nvfp4 (e2m1 x e2m1 block-scaled, fp32 accumulate)", "data": "synthetic",
            "config": {"workload": w["name"], "T": T, "H": H, "E": E, "topk": k, "I": I, "seed": w["seed"],
                       "four_six": four_six, "routed_rows": R, "padded_rows": R_pad,
                       "gemm_tflop_per_step": flops / 1e12,
                       "l2": "working set ~1 GB > 129 MB L2; no flush between steps; components rotate input sets > 2x L2",
                       "parallelism": f"replicas x{world}"},
            "roofline": roof, "mma_ceiling": ceiling,
            "hbm_write": {"gbs": P["hbm_write_gbs"], "source": P["hbm_write_source"]}, "stages": stages, "components": components, "e2e": e2e,
            "step_with_h_quantized_in_gemm1_ms": fused_h_ms, "second_record": second,
            "gpu_launches": KERNELS_PER_STEP * K, "clocks": clk}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, x_bits, ids)
    if rank == 0:
        print(json.dumps(line), flush=True)


def layer_record(bsq, synth, w, dev, P, steps=10, warmup=3):
    """Step time and per-stage breakdown of one MoE layer workload `w` (the
    second record of the bench line): inputs and weights generated on the
    device, `steps` forwards timed back to back with CUDA events, then the
    same number with events at the stage boundaries."""
    import torch
    T, H, I, E, k = w["T"], w["H"], w["I"], w["E"], w["k"]
    four_six = w.get("four_six", False)
    x = torch.from_numpy(synth.normal((T, H), seed=w["seed"]).view(np.int16)).view(torch.bfloat16).to(dev)
    ids, wts = synth.topk_routing(T, E, k, seed=w["seed"], zipf_s=w.get("zipf"))
    ids_d, wts_d = torch.from_numpy(ids).to(dev), torch.from_numpy(wts).to(dev)
    wb = synth.device_normal_bf16((E, 2 * I, H), seed=w["w_seed_gu"], std=0.02, device=dev)
    wgu = bsq.quantize_nvfp4_per_expert(wb)
    del wb
    wb = synth.device_normal_bf16((E, H, I), seed=w["w_seed_d"], std=0.02, device=dev)
    wd = bsq.quantize_nvfp4_per_expert(wb)
    del wb
    ws = torch.empty(bsq.moe_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=dev)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def fwd():
        bsq.moe_expert_forward(x, ids_d, wts_d, wgu, wd, I, four_six=four_six, workspace=ws, y=y, dev_status=status)

    for _ in range(warmup):
        fwd()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fwd()
    e1.record()
    torch.cuda.synchronize()
    ms_step = e0.elapsed_time(e1) / steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(steps)]
    for row in ev:  # torch creates an event's CUDA handle at its first record
        for e in row:
            e.record()
    torch.cuda.synchronize()
    for i in range(steps):
        bsq.set_stage_events(ev[i])
        fwd()
    bsq.set_stage_events(None)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    f1, f2 = gemm_flops(w)
    R = T * k
    L = bsq.moe_workspace_layout(T, H, I, E, k)
    R_pad = int(ws[L.offsets + 4 * E:L.offsets + 4 * (E + 1)].view(torch.int32).item())
    stages = stage_table(ev, w, R_pad, P)
    del x, ids_d, wts_d, wgu, wd, ws, y
    torch.cuda.empty_cache()
    return {"workload": w["name"], "metric": METRIC, "value": (f1 + f2) / (ms_step * 1e-3) / 1e12,
            "unit": "TFLOP/s", "ms_per_step": ms_step, "steps": steps, "warmup": warmup, "four_six": four_six,
            "routed_rows": R, "padded_rows": R_pad, "gemm_tflop_per_step": (f1 + f2) / 1e12, "stages": stages}


def time_rotating(launch, nsets, iters):
    """Per-launch device time of `launch(i)` for i = 0 .. iters-1, enqueued back
    to back between one pair of CUDA events on the current stream.  launch(i)
    uses buffer set i % nsets; the sets together exceed twice the 129 MB L2,
    so every launch finds its inputs evicted (no flush kernel is needed)."""
    import torch
    for i in range(2 * nsets):  # warm-up
        launch(i)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for i in range(iters):
        launch(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def backward_gemm_components(bsq, dev, P):
    """The MXFP8 grouped GEMM of the backward pass through the C ABI: the down
    projection's data gradient on the Qwen3-shaped layer (dh = dout . W_d over
    128 expert segments of 1024 / 1152 rows: M = 139264, K = H = 2048,
    N = I = 768, bf16 out), random finite E4M3 codes and E8M0 scales around 1,
    two input/output sets (1.4 GB) rotated."""
    import torch
    L = bsq.load()
    st = torch.cuda.current_stream(dev).cuda_stream
    E, K, N = 128, 2048, 768
    counts = [1024 if e % 2 == 0 else 1152 for e in range(E)]
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device=dev)
    M = int(sum(counts))
    g = torch.Generator(device=dev).manual_seed(13)

    def codes(*shape):
        c = torch.randint(0, 0x7E, shape, dtype=torch.uint8, device=dev, generator=g)
        return c | (torch.randint(0, 2, shape, dtype=torch.uint8, device=dev, generator=g) << 7)

    def sfs(rows):
        return torch.randint(120, 135, (bsq.sf_swizzled_bytes(rows, K // 32),), dtype=torch.uint8, device=dev,
                             generator=g)

    ones_m = torch.ones(M, dtype=torch.float32, device=dev)
    ones_e = torch.ones(E, dtype=torch.float32, device=dev)
    n = 2
    sets = [(codes(M, K), sfs(M), codes(E, N, K), sfs(E * N), torch.empty(M, N, dtype=torch.bfloat16, device=dev))
            for _ in range(n)]

    def mm(i):
        a, asf, b, bsf, out = sets[i % n]
        L.grouped_expert_gemm_mxfp8(a.data_ptr(), asf.data_ptr(), ones_m.data_ptr(), offsets.data_ptr(), E, M, K, N,
                                    b.data_ptr(), bsf.data_ptr(), ones_e.data_ptr(), bsq.EPI_BF16, out.data_ptr(), N,
                                    bsq.SF_SWIZZLED, None, st)

    us = time_rotating(mm, n, 10 * n) * 1e3
    flop = 2.0 * M * N * K
    del sets
    return {"mxfp8_gemm_dgrad_qwen3": {"us": us, "tflop": flop / 1e12, "tflops": flop / (us * 1e-6) / 1e12,
                                       "frac_of_fp8_peak": flop / (us * 1e-6) / 1e12 / P["fp8_tflops"],
                                       "fp8_peak_source": P["fp8_source"],
                                       "shape": "M=139264 (128 experts) K=2048 N=768, bf16 out", "sets": n}}


def quantizer_components(bsq, synth, dev, P):
    """The standalone bandwidth-bound kernels through the C ABI, rotating over
    input/output sets larger than L2 together (each launch starts cold)."""
    import torch
    L = bsq.load()
    st = torch.cuda.current_stream(dev).cuda_stream
    l2_twice = 2 * 129 * (1 << 20)
    out = {}

    def record(name, us, b, nsets):
        out[name] = {"us": us, "bytes": b, "gbs": b / (us * 1e-6) / 1e9, "frac_of_hbm": b / (us * 1e-6) / 1e9 / P["hbm_gbs"],
                     "sets": nsets}

    # MXFP8 row + column copies, 16384 x 2048, row std 10^U(-3,2)
    b = 16384 * 2048 * 2 + 2 * (16384 * 2048 + 16384 * 64)
    n = -(-l2_twice // b) + 1
    xm = torch.from_numpy(synth.rows_log_uniform_std(16384, 2048, seed=2).view(np.int16)).to(dev).view(torch.bfloat16)
    sets = [(xm.clone(), torch.empty(16384, 2048, dtype=torch.uint8, device=dev),
             torch.empty(16384, 64, dtype=torch.uint8, device=dev), torch.empty(2048, 16384, dtype=torch.uint8, device=dev),
             torch.empty(2048, 512, dtype=torch.uint8, device=dev)) for _ in range(n)]

    def mx(i):
        x, rc, rs, cc, cs = sets[i % n]
        L.quantize_mxfp8_rowcol(x.data_ptr(), 16384, 2048, 2048, rc.data_ptr(), rs.data_ptr(), cc.data_ptr(),
                                cs.data_ptr(), 0, None, st)

    record("mxfp8_rowcol_16384x2048", time_rotating(mx, n, 10 * n) * 1e3, b, n)
    del sets
    # NVFP4 per-token, 16384 x 2048 (swizzled SF)
    b = 16384 * 2048 * 2 + 16384 * (1024 + 128 + 4)
    n = -(-l2_twice // b) + 1
    xq = torch.from_numpy(synth.normal((16384, 2048), seed=3).view(np.int16)).to(dev).view(torch.bfloat16)
    sets = [(xq.clone(), torch.empty(16384, 1024, dtype=torch.uint8, device=dev),
             torch.empty(16384 * 128, dtype=torch.uint8, device=dev), torch.empty(16384, dtype=torch.float32, device=dev))
            for _ in range(n)]

    def nv(i):
        x, codes, sf, t = sets[i % n]
        L.quantize_nvfp4_per_token(x.data_ptr(), 16384, 2048, 2048, codes.data_ptr(), sf.data_ptr(), t.data_ptr(),
                                   bsq.SF_SWIZZLED, None, st)

    record("nvfp4_per_token_16384x2048", time_rotating(nv, n, 10 * n) * 1e3, b, n)

    def nr(i):
        x, codes, sf, t = sets[i % n]
        L.quantize_nvfp4_rht(x.data_ptr(), 16384, 2048, 2048, 7, codes.data_ptr(), sf.data_ptr(), t.data_ptr(),
                             bsq.SF_SWIZZLED, None, st)

    # the same with the 32-point random Hadamard transform in front (same bytes)
    record("nvfp4_rht_16384x2048", time_rotating(nr, n, 10 * n) * 1e3, b, n)
    del sets
    # BF16 dequantization of NVFP4 (the dequantized backward's operands), 16384 x 2048, swizzled SF
    b = 16384 * (1024 + 128 + 4) + 16384 * 2048 * 2
    n = -(-l2_twice // b) + 1
    c0, s0, t0 = bsq.quantize_nvfp4_per_token(xq, swizzled=True)
    sets = [(c0.clone(), s0.clone(), t0.clone(), torch.empty(16384, 2048, dtype=torch.bfloat16, device=dev))
            for _ in range(n)]

    def dq(i):
        c_, s_, t_, y_ = sets[i % n]
        L.dequantize_nvfp4(c_.data_ptr(), s_.data_ptr(), t_.data_ptr(), 16384, 2048, 1, y_.data_ptr(), 2048,
                           bsq.SF_SWIZZLED, None, st)

    record("dequant_nvfp4_16384x2048", time_rotating(dq, n, 10 * n) * 1e3, b, n)
    del sets
    # 2-D NVFP4 (16 x 16 tiles, per-tensor scale), both operand orientations, 16384 x 2048; the
    # tensor-maximum pre-pass re-reads x (from L2 when it fits) and is not counted as algorithmic
    b = 16384 * 2048 * 2 + 2 * (16384 * 1024 + 1024 * 128) + 4
    n = -(-l2_twice // b) + 1
    sets = [(xq.clone(), torch.empty(16384, 1024, dtype=torch.uint8, device=dev),
             torch.empty(1024, 128, dtype=torch.uint8, device=dev), torch.empty(2048, 8192, dtype=torch.uint8, device=dev),
             torch.empty(128, 1024, dtype=torch.uint8, device=dev), torch.empty(1, dtype=torch.float32, device=dev))
            for _ in range(n)]

    def q2(i):
        x_, c_, s_, ct_, st_, t_ = sets[i % n]
        L.quantize_nvfp4_2d(x_.data_ptr(), 16384, 2048, c_.data_ptr(), s_.data_ptr(), ct_.data_ptr(), st_.data_ptr(),
                            t_.data_ptr(), 0, None, st)

    record("nvfp4_2d_16384x2048", time_rotating(q2, n, 10 * n) * 1e3, b, n)
    del sets
    # requant with Philox SR (and round-to-nearest), both targets, 16384 x 2048 and 16384 x 768
    for K in (2048, 768):
        b = (16384 * K // 2 + 16384 * K // 16 + 16384 * 4) + (K * 8192 + K * 1024 + K * 4) + (K * 16384 + K * 512)
        n = -(-l2_twice // b) + 1
        xr = synth.normal_with_outliers(16384, K, seed=7)
        c, s, tt = bsq.quantize_nvfp4_per_token(torch.from_numpy(xr.view(np.int16)).to(dev).view(torch.bfloat16),
                                                swizzled=True)
        wsb = bsq.requant_workspace_size(16384, K)
        sets = [(c.clone(), s.clone(), tt.clone(), torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev),
                 torch.empty(K, 8192, dtype=torch.uint8, device=dev), torch.empty(K * 1024, dtype=torch.uint8, device=dev),
                 torch.empty(K, dtype=torch.float32, device=dev), torch.empty(K, 16384, dtype=torch.uint8, device=dev),
                 torch.empty(((K + 127) // 128 * 128) * 512, dtype=torch.uint8, device=dev)) for _ in range(n)]
        for sr in (True, False):
            flags = bsq.SF_SWIZZLED | (bsq.STOCHASTIC if sr else 0)

            def rq(i):
                cc_, ss_, tt_, ws, nc, ns, nt, mc, ms = sets[i % n]
                L.requant_transpose_sr(cc_.data_ptr(), ss_.data_ptr(), tt_.data_ptr(), 16384, K, nc.data_ptr(),
                                       ns.data_ptr(), nt.data_ptr(), mc.data_ptr(), ms.data_ptr(), 7, ws.data_ptr(),
                                       wsb, flags, None, st)

            record(f"requant_{'sr' if sr else 'rne'}_16384x{K}", time_rotating(rq, n, 10 * n) * 1e3, b, n)
        del sets
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="qwen3")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-components", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, w, rank, world)
    else:
        run_ours(args, w, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
