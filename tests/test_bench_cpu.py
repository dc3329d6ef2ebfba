"""Host arithmetic of bench.py that turns stage times into rates, checked on
CPU with stand-in events: the algorithmic bytes of the forward's
data-moving stages and the HBM floor (the longer of all bytes at the copy
rate and the written bytes at the write-only rate)."""
import os
import sys

import pytest

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


class _Ev:
    """Stands in for a recorded torch.cuda.Event: elapsed_time in ms."""

    def __init__(self, t_ms):
        self.t = t_ms

    def elapsed_time(self, other):
        return other.t - self.t


QWEN3 = bench.WORKLOADS["qwen3"]


def test_stage_traffic_of_the_qwen3_layer():
    R_pad = 139264
    tr = bench.stage_traffic(QWEN3, R_pad)
    T, H, I, E, k = 16384, 2048, 768, 128, 8
    R = T * k
    # x read once; each routed copy: H/2 code bytes, H/16 scale bytes, one fp32 scale
    assert tr["quantize_scatter"] == (T * H * 2, R * (1024 + 128 + 4))
    # h (bf16) read; its codes, scale bytes and fp32 scale written
    assert tr["quantize_h"] == (R_pad * I * 2, R_pad * (384 + 48 + 4))
    # GEMM2: A codes + scales + row scales, the experts' weights and their scales; bf16 out
    assert tr["gemm2"] == (R_pad * (384 + 48 + 4) + E * H * (384 + 48), R_pad * H * 2)
    # combine: the k rows of every token (+ its slot and weight), y written
    assert tr["combine"] == (R * H * 2 + R * 8, T * H * 2)


def test_stage_table_rates_and_hbm_floor():
    R_pad = 139264
    P = {"hbm_gbs": 6800.0, "hbm_write_gbs": 3000.0, "fp4_tflops": 9000.0}
    # stage s lasts 0.01 * (s + 1) ms, the same in both event rows
    bounds = [0.0]
    for s in range(6):
        bounds.append(bounds[-1] + 0.01 * (s + 1))
    ev = [[_Ev(b) for b in bounds] for _ in range(2)]
    st = bench.stage_table(ev, QWEN3, R_pad, P)
    assert list(st) == bench.STAGES
    for s, n in enumerate(bench.STAGES):
        assert st[n]["ms"] == pytest.approx(0.01 * (s + 1))
    tr = bench.stage_traffic(QWEN3, R_pad)
    for n, (rd, wr) in tr.items():
        ms = st[n]["ms"]
        floor_ms = max((rd + wr) / 6800e9, wr / 3000e9) * 1e3
        assert st[n]["hbm_floor_ms"] == pytest.approx(floor_ms)
        assert st[n]["frac_of_hbm_floor"] == pytest.approx(floor_ms / ms)
        if n != "gemm2":
            assert st[n]["gbs"] == pytest.approx((rd + wr) / (ms * 1e-3) / 1e9)
            assert st[n]["frac_of_hbm"] == pytest.approx(st[n]["gbs"] / 6800.0)
    # with a write rate below the copy rate, the write-heavy stages are floored by their writes
    rd, wr = tr["quantize_scatter"]
    assert wr / 3000e9 > (rd + wr) / 6800e9
    f1, f2 = bench.gemm_flops(QWEN3)
    assert st["gemm1_swiglu"]["tflops"] == pytest.approx(f1 / (0.03e-3) / 1e12)
    assert st["gemm2"]["tflops"] == pytest.approx(f2 / (0.05e-3) / 1e12)
    assert "hbm_floor_ms" not in st["route"] and "gbs" not in st["gemm1_swiglu"]


def test_stage_table_without_a_write_rate_reports_no_floor():
    ev = [[_Ev(0.01 * i) for i in range(7)]]
    st = bench.stage_table(ev, QWEN3, 139264, {"hbm_gbs": 6800.0, "fp4_tflops": 9000.0})
    assert all("hbm_floor_ms" not in d for d in st.values())
    assert st["combine"]["frac_of_hbm"] > 0
