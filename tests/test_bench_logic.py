"""Host-side logic of bench.py: algorithmic work accounting and the clock parser (no GPU)."""
import os

import pytest

import bench
import moe_inputs as mi


@pytest.mark.parametrize("name", list(mi.CONFIGS))
def test_kernel_flops_add_up_to_layer_flops(name):
    cfg = mi.CONFIGS[name]
    w = bench.kernel_work(cfg)
    kernels = [k for k in w if k.startswith(("gemm_", "proj_", "wgrad_"))]
    assert sum(w[k]["flops"] for k in kernels) == bench.step_flops(cfg)
    if name in ("gptoss20b", "gptoss120b_skew"):
        for k in bench.GEMM_KERNELS:
            assert w[k]["bound"] == "tensor"
    for k in kernels:
        if k.startswith(("proj_", "wgrad_")):
            assert w[k]["bound"] == "hbm"


def test_slot_rows_are_bf16_in_the_byte_model():
    # the forward's O rows and the backward's dX rows are both one bf16 row per routed slot,
    # so the two combines move the same bytes, and the gate_up backward writes N*H*2 bytes
    cfg = mi.CONFIGS["gptoss20b"]
    w = bench.kernel_work(cfg)
    assert w["combine_dx"]["bytes"] == w["combine_y"]["bytes"]
    N, H, I, E, r = cfg.T * cfg.k, cfg.H, cfg.I, cfg.E, cfg.r
    assert w["gemm_gate_up_bwd"]["bytes"] == 2 * (N * 2 * I + E * H * 2 * I + E * r * H + N * 16 + N * H)
    assert abs(w["gemm_gate_up_bwd"]["bytes"] / 1e9 - 1.348) < 1e-3


def test_step_flops_matches_closed_form_for_gptoss20b():
    cfg = mi.CONFIGS["gptoss20b"]
    N = cfg.T * cfg.k
    assert bench.step_flops(cfg) == N * (12 * 2880 * 2880 + 12 * 2880 * 16 + 18 * 2880 * 16)
    assert abs(bench.step_flops(cfg) / 1e12 - 1.6534) < 1e-3


def test_clock_sampler_parses_nvidia_smi_csv(tmp_path, monkeypatch):
    s = bench.ClockSampler(0)
    p = tmp_path / "c.csv"
    p.write_text("0, 1980, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Active\n"
                 "0, 2000, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                 "0, 1990, 2070, 930.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")

    class FakeProc:
        def terminate(self): pass
        def wait(self, timeout=None): return 0
        def kill(self): pass
    s.proc, s.path = FakeProc(), str(p)
    monkeypatch.setattr(bench.time, "sleep", lambda _: None)
    out = s.stop()
    assert out["sm_mhz"] == 1990 and out["sm_max_mhz"] == 2070 and out["reasons"] == ["sw_power_cap"]
    assert not os.path.exists(p)


def test_load_peaks_reads_measured_file():
    pk = bench.load_peaks()
    assert pk["hbm_gbs"] > 1000 and pk["bf16_tflops"] > 100


def test_routing_summary_shows_the_skew():
    import bench
    cfg = mi.CONFIGS["gptoss120b_skew"]
    idx, _ = mi.make_routing(cfg, 0)
    r = bench.routing_summary(idx, cfg.E)
    assert sum(r["counts"]) == cfg.T * cfg.k and len(r["counts"]) == cfg.E
    assert r["zero_experts"] > 0 and r["above_10x_mean"] > 0      # many empty experts, a few hot ones
    flat = mi.CONFIGS["gptoss20b"]
    r2 = bench.routing_summary(mi.make_routing(flat, 0)[0], flat.E)
    assert r2["zero_experts"] == 0 and r2["above_10x_mean"] == 0


def test_tensor_peak_is_the_burst_figure_at_full_clock():
    """Kernels timed inside a few-millisecond step at the maximum SM clock are held against the
    burst bf16 peak; a run whose median clock fell more than 5 % below the maximum (a power cap
    that bit, or a clock lock) against the sustained one; no clock record: sustained."""
    peaks = dict(hbm_gbs=6690.0, bf16_tflops=1924.2, bf16_tflops_sustained=1735.4, source="measured")
    p, src = bench.tensor_peak(peaks, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0})
    assert p == 1924.2 and "burst" in src and "2070" in src
    p, _ = bench.tensor_peak(peaks, {"sm_mhz": 1976.0, "sm_max_mhz": 2070.0})
    assert p == 1924.2
    p, src = bench.tensor_peak(peaks, {"sm_mhz": 1900.0, "sm_max_mhz": 2070.0})
    assert p == 1735.4 and "sustained" in src
    p, _ = bench.tensor_peak(peaks, {"sm_mhz": None, "sm_max_mhz": None})
    assert p == 1735.4


def test_routing_summary_shows_the_skewed_histogram():
    """The skewed workload's routing: many experts without rows and a few above ten times
    the mean, as the bench line reports them."""
    cfg = mi.CONFIGS["gptoss120b_skew"]
    idx, _ = mi.make_routing(cfg, 0)
    s = bench.routing_summary(idx, cfg.E)
    assert s["zero_experts"] >= 10 and s["above_10x_mean"] >= 1
    assert sum(s["counts"]) == cfg.T * cfg.k and s["max"] == max(s["counts"])
