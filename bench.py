"""Benchmark of the MoE-LoRA expert layer (route + forward + backward) on GB300.

One step = moe_route + moe_lora_fwd + moe_lora_bwd over one synthetic batch of
the GPT-OSS-20B-shaped layer (T=4096, H=2880, E=32, top-4, I=2880, LoRA r=16)
unless --config says otherwise.  Prints ONE JSON line (rank 0).

  value        tokens/s of the whole job, device-timed (CUDA events around every
               step, inputs resident in HBM, L2 flushed between steps)
  e2e          the same metric with every step's inputs copied from pinned host
               memory and its results (y, dx, LoRA gradients) copied back inside
               one timed span; two step slots on three streams, so copies of
               neighbouring steps overlap a step's compute (no L2 flush there:
               the weights alone exceed L2)
  roofline     the dominant kernel (largest share of the step), its algorithmic
               flops (or bytes) per launch over its event-timed duration (CUDA
               events around each library launch, in a second timed pass of the
               same steps: they cost ~2 % of a step, so the value pass runs
               without them)
  graph_ms_per_step  the same step replayed from a captured CUDA graph (launch
               gaps removed), for information
  gemm         all grouped-GEMM kernels together: algorithmic TFLOP/s and the
               fraction of the measured dense bf16 peak (the burst figure when the
               median SM clock of the run stayed within 5 % of its maximum, else the
               sustained one; the other is kept beside it)
  other_configs  the Qwen3-30B-A3B, skewed GPT-OSS-120B and DeepSeek-V3 shapes, a
               short run each (10 steps): ms/step, tokens/s, grouped-GEMM TFLOP/s,
               the dominant kernel against its roofline, the routing histogram, and
               the FP8- and NF4-base steps of the DeepSeek-V3 shape
  cpu_baseline the CPU oracle timed on a bounded token sample (rank 0, N=1): route,
               forward and backward separately, the threads used, and the tiny layer
               on one thread

--impl reference times the CPU oracle (the only reference this layer has) on
the host cores, on bounded token samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import moe_inputs as mi  # noqa: E402

METRIC = "MoE-layer fwd+bwd tokens/s; grouped-GEMM TFLOP/s as % of GB300 BF16 peak"
UNIT = "tokens/s"
GEMM_KERNELS = ("gemm_gate_up_fwd", "gemm_down_fwd", "gemm_down_bwd", "gemm_gate_up_bwd")


# ----------------------------------------------------------------------------- algorithmic work
def kernel_work(cfg: mi.MoEConfig, ridge: float | None = None) -> dict:
    """Algorithmic flops and HBM bytes of one launch of each kernel (bf16 = 2 B).

    N = T*k routed rows.  GEMM flops count the base and the LoRA product the
    kernel performs; bytes count each operand once (weights of all experts).
    A kernel is tensor-bound when its flops per byte reach the ridge point
    (dense bf16 peak / HBM bandwidth), else HBM-bound."""
    if ridge is None:
        pk = load_peaks()
        ridge = pk["bf16_tflops_sustained"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    T, H, I, E, k, r = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r
    N = T * k
    rp = 16 if r <= 16 else (32 if r <= 32 else 64)
    b = 2
    w = {
        "gemm_gate_up_fwd": dict(flops=2 * N * H * 2 * I + 2 * N * r * 2 * I,
                                 bytes=b * (N * H + E * H * 2 * I + E * r * 2 * I + N * rp + N * 2 * I + N * I)),
        "gemm_down_fwd": dict(flops=2 * N * I * H + 2 * N * r * H,
                              bytes=b * (N * I + E * I * H + E * r * H + N * rp + N * H)),
        "gemm_down_bwd": dict(flops=2 * N * H * I + 2 * N * r * I,
                              bytes=b * (N * H + E * I * H + E * r * I + N * rp + N * 2 * I + N * 2 * I)),
        "gemm_gate_up_bwd": dict(flops=2 * N * 2 * I * H + 2 * N * r * H,
                                 bytes=b * (N * 2 * I + E * H * 2 * I + E * r * H + N * rp + N * H)),
        "gather_x": dict(flops=0, bytes=b * (T * H + N * H) + 4 * N),
        "gather_dy": dict(flops=N * H, bytes=b * (T * H + N * H) + 8 * N),
        "proj_xa": dict(flops=2 * N * H * r, bytes=b * (N * H + E * r * H + N * rp)),
        "proj_ha": dict(flops=2 * N * I * r, bytes=b * (N * I + E * r * I + N * rp)),
        "proj_g": dict(flops=2 * N * H * r, bytes=b * (N * H + E * r * H + N * rp)),
        "proj_gg": dict(flops=2 * N * 2 * I * r, bytes=b * (N * 2 * I + E * r * 2 * I + N * rp)),
        "combine_y": dict(flops=N * H, bytes=b * N * H + b * T * H + 4 * N),
        "combine_dx": dict(flops=N * H, bytes=b * N * H + b * T * H + 4 * N),
        "wgrad_down": dict(flops=2 * N * r * I + 2 * N * r * H,
                           bytes=b * (2 * N * rp + N * I + N * H + E * r * I + E * r * H)),
        "wgrad_gate_up": dict(flops=2 * N * r * H + 2 * N * r * 2 * I,
                              bytes=b * (2 * N * rp + N * H + N * 2 * I + E * r * H + E * r * 2 * I)),
        "route": dict(flops=0, bytes=N * (8 + 4) * 2 + N * 12 + 8 * (E + 1)),
    }
    for v in w.values():
        v["bound"] = "tensor" if v["flops"] >= ridge * v["bytes"] else "hbm"
    return w


# DRAM bytes (read + write) per launch from ncu captures of the current kernels
# (profiles/), keyed by (workload, kernel); None where no capture of the current code exists.
MEASURED_TRAFFIC = {
    ("gptoss20b", "gemm_gate_up_fwd"): 1.1715e9 + 0.2616e9,
    ("gptoss20b", "gemm_down_fwd"): 0.6333e9 + 0.0799e9,
    ("gptoss20b", "gemm_down_bwd"): 0.8380e9 + 0.1637e9,
    ("gptoss20b", "gemm_gate_up_bwd"): 1.3208e9 + 0.0864e9,
}


def step_flops(cfg: mi.MoEConfig) -> int:
    """Algorithmic fwd+bwd flops of the layer: N (12 H I + 12 H r + 18 I r)."""
    N = cfg.T * cfg.k
    return N * (12 * cfg.H * cfg.I + 12 * cfg.H * cfg.r + 18 * cfg.I * cfg.r)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=p["hbm_gbs"], bf16_tflops=p["bf16_tflops"],
                    bf16_tflops_sustained=p.get("bf16_tflops_sustained", p["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def tensor_peak(peaks: dict, clk: dict) -> tuple[float, str]:
    """Dense bf16 peak to hold a kernel against: the burst figure (a short GEMM at full
    clock) when the run's median SM clock under load stayed within 5 % of the maximum, as
    it does for the few-millisecond steps timed here; the sustained figure (a seconds-long
    GEMM loop that settles under the power cap) otherwise."""
    mhz, mx = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    if mhz is not None and mx and mhz >= 0.95 * mx:
        return peaks["bf16_tflops"], f"{peaks['source']} bf16 burst (median SM clock {mhz:.0f} of {mx:.0f} MHz)"
    return peaks["bf16_tflops_sustained"], f"{peaks['source']} bf16 sustained (median SM clock {mhz} of {mx} MHz)"


# ----------------------------------------------------------------------------- ranks
def max_over_ranks(value: float, device=None) -> float:
    """Largest `value` over all ranks (identity without torch.distributed): the job's
    time is its slowest replica's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_replica_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job tokens/s of `world` independent replicas (weak scaling): all replicas'
    tokens over the slowest replica's time."""
    return tokens_per_replica_step * steps * world / (max_ms / 1e3)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None, "samples": len(rows), "reasons": reasons}


# ----------------------------------------------------------------------------- CPU oracle timing
def oracle_sample_step(cfg, idx, w, x_cpu, dy_cpu, wts_cpu, S: int, parts: dict | None = None) -> float:
    """Route the full batch and run forward + backward of the oracle on the first
    S tokens as a batch of their own; returns seconds (and, in `parts`, the seconds
    of the route, the forward and the backward)."""
    from oracle import moe_oracle as orc
    t0 = time.perf_counter()
    orc.route(idx, cfg.E)
    t1 = time.perf_counter()
    sub_idx, sub_w = idx[:S], w[:S]
    orc.lora_fwd(x_cpu[:S], sub_idx, sub_w, *wts_cpu, cfg.scale)
    t2 = time.perf_counter()
    orc.lora_bwd(dy_cpu[:S], x_cpu[:S], sub_idx, sub_w, *wts_cpu, cfg.scale)
    t3 = time.perf_counter()
    if parts is not None:
        parts.update(route_s=t1 - t0, fwd_s=t2 - t1, bwd_s=t3 - t2)
    return t3 - t0


def oracle_threads() -> dict:
    """Threads the oracle runs on: numpy's BLAS (its float64 matmuls) and torch's
    intra-op pool (the bf16 -> float64 conversions)."""
    import torch
    out = {"torch_threads": torch.get_num_threads(), "blas_threads": None}
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        out["blas_threads"] = max(n) if n else None
    except ImportError:
        env = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
        out["blas_threads"] = int(env) if env else os.cpu_count()
    return out


def tiny_oracle_one_thread(seed: int = 0, reps: int = 5) -> dict:
    """The tiny layer (T = 64) through the oracle in a child process pinned to one
    thread (BLAS and torch): median seconds of route, forward and backward."""
    code = (
        "import json,os,sys,time,statistics;sys.path.insert(0,%r);import torch;torch.set_num_threads(1);"
        "import moe_inputs as mi;from oracle import moe_oracle as orc;cfg=mi.CONFIGS['tiny'];"
        "idx,w=mi.make_routing(cfg,%d);ts=mi.make_tensors(cfg,%d,'cpu');"
        "wts=[ts[n] for n in ('W_gu','A_gu','B_gu','W_d','A_d','B_d')];r=[]\n"
        "for _ in range(%d):\n"
        " t0=time.perf_counter();orc.route(idx,cfg.E);t1=time.perf_counter();"
        "orc.lora_fwd(ts['x'],idx,w,*wts,cfg.scale);t2=time.perf_counter();"
        "orc.lora_bwd(ts['dy'],ts['x'],idx,w,*wts,cfg.scale);t3=time.perf_counter();r.append((t1-t0,t2-t1,t3-t2))\n"
        "m=[statistics.median(v) for v in zip(*r)];"
        "print(json.dumps({'route_s':m[0],'fwd_s':m[1],'bwd_s':m[2],'tokens_per_s':cfg.T/sum(m)}))"
    ) % (ROOT, seed, seed, reps)
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=300)
        return json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else {"error": r.stderr[-300:]}
    except (subprocess.TimeoutExpired, IndexError, ValueError) as exc:
        return {"error": str(exc)}


def cpu_baseline(cfg, idx, w, x_cpu, dy_cpu, wts_cpu, budget_s: float = 25.0) -> dict:
    # two-point calibration: a fixed part (routing all tokens, per-expert weight merges)
    # plus a per-token part
    t2 = oracle_sample_step(cfg, idx, w, x_cpu, dy_cpu, wts_cpu, 2)
    t8 = oracle_sample_step(cfg, idx, w, x_cpu, dy_cpu, wts_cpu, 8)
    slope = max((t8 - t2) / 6.0, 1e-6)
    S = int(max(8, min(cfg.T, 8 + (budget_s - t8) / slope)))
    parts = {}
    t = oracle_sample_step(cfg, idx, w, x_cpu, dy_cpu, wts_cpu, S, parts)
    return {"value": S / t, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle", **oracle_threads(),
            "sample": f"route of all {cfg.T} tokens + fp64 forward and backward of the first {S} tokens "
                      f"as a batch ({t:.1f} s)",
            "route_s": parts["route_s"], "fwd_s": parts["fwd_s"], "bwd_s": parts["bwd_s"],
            "route_tokens_per_s": cfg.T / parts["route_s"], "fwd_bwd_tokens_per_s": S / (parts["fwd_s"] + parts["bwd_s"]),
            "tiny_layer_1_thread": tiny_oracle_one_thread()}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, cfg):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch
    idx, w = mi.make_routing(cfg, args.seed)
    ts = mi.make_tensors(cfg, args.seed, "cuda" if torch.cuda.is_available() else "cpu")
    wts = [ts[n].cpu() for n in ("W_gu", "A_gu", "B_gu", "W_d", "A_d", "B_d")]
    x_cpu, dy_cpu = ts["x"].cpu(), ts["dy"].cpu()
    del ts
    budget = 150.0 / max(1, args.steps + args.warmup)
    t2 = oracle_sample_step(cfg, idx, w, x_cpu, dy_cpu, wts, 1)
    S = int(max(1, min(cfg.T, budget / max(t2, 1e-6))))
    for _ in range(args.warmup):
        oracle_sample_step(cfg, idx, w, x_cpu, dy_cpu, wts, S)
    times = [oracle_sample_step(cfg, idx, w, x_cpu, dy_cpu, wts, S) for _ in range(args.steps)]
    total = sum(times)
    value = S * args.steps / total
    sample = f"route of all {cfg.T} tokens + fp64 forward and backward of the first {S} tokens per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(cfg),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_dict(cfg):
    return {"workload": f"{cfg.name}: T={cfg.T} H={cfg.H} E={cfg.E} top-{cfg.k} I={cfg.I} LoRA r={cfg.r} "
                        f"alpha={cfg.alpha:g}" + (f" zipf={cfg.zipf_s}" if cfg.zipf_s else ""),
            "T": cfg.T, "H": cfg.H, "E": cfg.E, "k": cfg.k, "I": cfg.I, "r": cfg.r,
            "l2": "flushed between steps (256 MiB write); inputs+weights also exceed L2"}


def routing_summary(idx, E: int) -> dict:
    """Expert row counts of the workload's routing (the skewed workload's histogram shows
    its empty experts and hot ones)."""
    counts = np.bincount(np.asarray(idx).reshape(-1), minlength=E)
    mean = counts.sum() / E
    out = {"min": int(counts.min()), "max": int(counts.max()), "mean": float(mean),
           "zero_experts": int((counts == 0).sum()), "above_10x_mean": int((counts > 10 * mean).sum())}
    if E <= 256:
        out["counts"] = counts.tolist()
    return out


# ----------------------------------------------------------------------------- quantised base weights
QUANT_KEYS = {"fp8": ("Wq", "s_"), "nf4": ("W4", "m_")}


def quant_measurement(cfg, layer, ts, t_idx, t_w, moe, dev, steps: int, flush, fmt: str) -> dict:
    """route + fwd + bwd with the expert base weights quantised (fmt "fp8": e4m3 codes +
    power-of-two column scales; "nf4": 4-bit NormalFloat codes + 64-element absmax
    scales), timed like the main loop."""
    import torch
    wq = moe.quantize_expert_weights(layer.w, fmt=fmt)
    q8 = moe.MoELoRALayer(layer.d, wq, dev)
    for _ in range(3):
        q8.step(t_idx, t_w, ts["x"], ts["dy"], with_topk_grad=False)
    torch.cuda.synchronize()
    moe.moe_timing_enable(True)
    per_step = []
    for _ in range(steps):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        q8.step(t_idx, t_w, ts["x"], ts["dy"], with_topk_grad=False)
        e.record()
        torch.cuda.synchronize()
        per_step.append(s.elapsed_time(e))
    moe.moe_timing_enable(False)
    kt = moe.moe_timing_read()
    assert int(q8.dev_status.item()) == 0
    gemm_ms = sum(kt[n][0] for n in GEMM_KERNELS if n in kt) / steps
    kernels = {n: round(v[0] / steps, 4) for n, v in kt.items() if n in GEMM_KERNELS}
    wbytes = sum(t.numel() * t.element_size() for n, t in wq.items() if n.startswith(QUANT_KEYS[fmt]))
    del q8, wq
    ms = sum(per_step)
    # the median beside the mean: a side line of few steps, where one slow step shows
    return {"ms_per_step": ms / steps, "median_ms_per_step": sorted(per_step)[steps // 2],
            "tokens_per_s": cfg.T * steps / (ms / 1e3), "gemm_ms_per_step": gemm_ms,
            "gemm_kernels_ms_per_step": kernels, "base_weight_bytes": wbytes, "steps": steps}


# ----------------------------------------------------------------------------- offload
def offload_measurement(cfg, layer, ts, t_idx, t_w, moe, dev, L: int, reps: int) -> dict:
    """Backward of an L-layer stack (shared weights) with the saved activations in
    pinned host memory, reloaded with two device buffers or one, against the same
    stack with every layer's activations resident."""
    import torch
    from moe_expert_dispatch_stable_gb300.offload import OffloadedMoEStack
    weights = [layer.w] * L
    routing = [(t_idx, t_w)] * L
    out = {"layers": L, "saved_bytes_per_layer": None}
    resident = [moe.MoELoRALayer(layer.d, layer.w, dev) for _ in range(L)]

    def once(fn):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e)

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        return statistics.median(once(fn) for _ in range(reps))

    def res_fwd():
        x = ts["x"]
        for l in range(L):
            resident[l].route(*routing[l])
            x = resident[l].forward(x)

    def res_bwd():
        g = ts["dy"]
        for l in range(L - 1, -1, -1):
            g = resident[l].backward(g, with_topk_grad=False)[0]
    res_fwd()
    out["bwd_ms_resident"] = timed(res_bwd)
    del resident
    # both stacks live at once and their repetitions alternate, so that the two reload
    # schedules see the same host-link conditions (it is shared with other work on the host)
    stacks = {name: OffloadedMoEStack(layer.d, weights, dev, buffers=nb) for name, nb in (("double", 2), ("single", 1))}
    for st in stacks.values():
        out["saved_bytes_per_layer"] = st.saved_bytes
        out["h2d_bytes_per_layer"] = st.transfer_bytes
        st.forward(ts["x"], routing)
        st.backward(ts["dy"])
    torch.cuda.synchronize()
    samples = {name: [] for name in stacks}
    for _ in range(reps):
        for name, st in stacks.items():
            samples[name].append(once(lambda: st.backward(ts["dy"])))
    for name in stacks:
        out[f"bwd_ms_{name}"] = statistics.median(samples[name])
    del stacks
    torch.cuda.empty_cache()
    out["h2d_gb_per_bwd"] = L * out["h2d_bytes_per_layer"] / 1e9
    return out


# ----------------------------------------------------------------------------- the other workloads
def workload_measurement(name: str, moe, dev, flush, steps: int, peaks: dict, seed: int, fp8: bool) -> dict:
    """A short run of another workload on the same line: route + fwd + bwd per step
    (CUDA events around each step, L2 flushed between steps), its grouped GEMMs against
    the dense bf16 peak, the dominant kernel against its roofline, and, with `fp8`, the
    same step with FP8 and with NF4 base weights.  The clocks of the main run decide burst or
    sustained peak; this short run sits right after it."""
    import torch
    cfg = mi.CONFIGS[name]
    idx, w = mi.make_routing(cfg, seed)
    ts = mi.make_tensors(cfg, seed, dev)
    layer = moe.MoELoRALayer(moe.Dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r, cfg.scale), ts, dev)
    t_idx, t_w = torch.from_numpy(idx).to(dev), torch.from_numpy(w).to(dev)

    def run(lay, timing: bool):
        for _ in range(3):
            lay.step(t_idx, t_w, ts["x"], ts["dy"], with_topk_grad=False)
        torch.cuda.synchronize()
        if timing:
            moe.moe_timing_enable(True)
        ms = []
        for _ in range(steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            lay.step(t_idx, t_w, ts["x"], ts["dy"], with_topk_grad=False)
            b.record()
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        if timing:
            moe.moe_timing_enable(False)
        assert int(lay.dev_status.item()) == 0, f"device status flag set ({name})"
        return sum(ms) / steps, (moe.moe_timing_read() if timing else None)

    step_ms, _ = run(layer, False)
    _, kt = run(layer, True)
    work = kernel_work(cfg)
    g_ms = sum(kt[n][0] for n in GEMM_KERNELS if n in kt) / steps
    g_fl = sum(work[n]["flops"] for n in GEMM_KERNELS)
    dom = max(kt, key=lambda n: kt[n][0])
    d_ms = kt[dom][0] / kt[dom][1]
    out = {"workload": config_dict(cfg)["workload"], "steps": steps, "ms_per_step": step_ms,
           "tokens_per_s": cfg.T / (step_ms / 1e3),
           "layer_tflops": step_flops(cfg) / (step_ms / 1e3) / 1e12,
           "gemm": {"ms_per_step": g_ms, "tflops": g_fl / (g_ms / 1e3) / 1e12,
                    "frac_of_bf16_burst": g_fl / (g_ms / 1e3) / 1e12 / peaks["bf16_tflops"],
                    "frac_of_bf16_sustained": g_fl / (g_ms / 1e3) / 1e12 / peaks["bf16_tflops_sustained"]},
           "dominant_kernel": {"kernel": dom, "ms_per_launch": d_ms, "bound": work[dom]["bound"],
                               "hbm_gbs": work[dom]["bytes"] / (d_ms / 1e3) / 1e9,
                               "frac_of_hbm": work[dom]["bytes"] / (d_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                               "tflops": work[dom]["flops"] / (d_ms / 1e3) / 1e12,
                               "frac_of_bf16_burst": work[dom]["flops"] / (d_ms / 1e3) / 1e12 / peaks["bf16_tflops"]},
           "kernels_ms_per_step": {n: round(v[0] / steps, 4) for n, v in sorted(kt.items(), key=lambda kv: -kv[1][0])},
           "routing": routing_summary(idx, cfg.E)}
    for fmt in ("fp8", "nf4") if fp8 else ():
        wq = moe.quantize_expert_weights(layer.w, fmt=fmt)
        lq = moe.MoELoRALayer(layer.d, wq, dev)
        f_ms, f_kt = run(lq, True)
        out[fmt + "_base"] = {"ms_per_step": f_ms, "tokens_per_s": cfg.T / (f_ms / 1e3),
                              "gemm_ms_per_step": sum(f_kt[n][0] for n in GEMM_KERNELS if n in f_kt) / steps,
                              "gemm_kernels_ms_per_step": {n: round(f_kt[n][0] / steps, 4) for n in GEMM_KERNELS
                                                           if n in f_kt}}
        del lq, wq
    del layer, ts
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------- GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="gptoss20b", choices=list(mi.CONFIGS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--breakdown", action="store_true", help="print per-kernel times to stderr")
    ap.add_argument("--no-offload", action="store_true", help="skip the offloaded-stack measurement")
    ap.add_argument("--no-fp8", action="store_true", help="skip the quantised-base-weight (FP8, NF4) measurements")
    ap.add_argument("--offload-layers", type=int, default=4)
    ap.add_argument("--other-steps", type=int, default=10,
                    help="timed steps of each other workload on the line (0: none)")
    ap.add_argument("--steps-only", action="store_true",
                    help="run the warm-up and timed steps of the layer, print the line's step time and exit "
                         "(a short command for profilers)")
    ap.add_argument("--base", default="bf16", choices=["bf16", "fp8", "nf4"],
                    help="with --steps-only: the expert base weights' format")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    cfg = mi.CONFIGS[args.config]
    if args.impl == "reference":
        run_reference(args, cfg)
        return

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    import moe_expert_dispatch_stable_gb300 as moe

    # inputs: weights shared by all replicas, activations per replica
    idx, w = mi.make_routing(cfg, args.seed + rank)
    ts = mi.make_tensors(cfg, args.seed, dev, names=("W_gu", "A_gu", "B_gu", "W_d", "A_d", "B_d"))
    ts.update(mi.make_tensors(cfg, args.seed + rank, dev, names=("x", "dy")))
    d = moe.Dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r, cfg.scale)
    if args.base != "bf16" and not args.steps_only:
        raise SystemExit("--base applies to --steps-only runs")
    layer = moe.MoELoRALayer(d, ts if args.base == "bf16" else moe.quantize_expert_weights(ts, fmt=args.base), dev)
    t_idx = torch.from_numpy(idx).to(dev)
    t_w = torch.from_numpy(w).to(dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        layer.step(t_idx, t_w, ts["x"], ts["dy"], with_topk_grad=False)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0, "device status flag set during warm-up"

    # ---- device-timed region: the public-API step, CUDA events around every step
    clocks = ClockSampler(local)
    clocks.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = moe.moe_launch_count()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        layer.step(t_idx, t_w, ts["x"], ts["dy"], with_topk_grad=False)
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    launches = moe.moe_launch_count() - launches0
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(sum(step_ms), dev)
    value = job_throughput(cfg.T, args.steps, world, total_ms)
    if args.steps_only:
        clocks.stop()
        assert int(layer.dev_status.item()) == 0, "device status flag set"
        if rank == 0:
            print(json.dumps({"steps_only": True, "config": config_dict(cfg), "base": args.base,
                              "ms_per_step": total_ms / args.steps,
                              "value": value, "unit": UNIT}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    # ---- per-kernel durations: a second timed pass of the same steps with the library's
    # CUDA events around each of its launches (on the caller's stream); they add ~2 % to
    # a step, so the pass above runs without them
    torch.cuda.synchronize()
    moe.moe_timing_enable(True)
    for i in range(args.steps):
        flush.zero_()
        layer.step(t_idx, t_w, ts["x"], ts["dy"], with_topk_grad=False)
    torch.cuda.synchronize()
    moe.moe_timing_enable(False)
    kt = moe.moe_timing_read()

    # ---- the same step replayed from a CUDA graph (for information: launch gaps)
    graph_ms = None
    try:
        gs = torch.cuda.Stream(dev)
        gs.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            layer.step(t_idx, t_w, ts["x"], ts["dy"], with_topk_grad=False)
        torch.cuda.synchronize()
        g_tot = 0.0
        for i in range(max(10, args.steps // 4)):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            g_tot += a.elapsed_time(b)
        graph_ms = g_tot / max(10, args.steps // 4)
        del g
    except RuntimeError as exc:                          # capture unsupported: report why
        graph_ms = f"unavailable: {exc}"

    # ---- end to end through host buffers: every step copies its inputs from pinned host
    # memory and its results (y, dx, LoRA gradients) back.  Two step slots (inputs and a
    # layer each) on three streams, so that step i+1's upload and step i-1's download run
    # while step i computes; one continuous timed span from the first upload to the last
    # download.  No L2 flush in this span: the weights alone (>= 1.6 GB) exceed L2.
    h_x = ts["x"].cpu().pin_memory(); h_dy = ts["dy"].cpu().pin_memory()
    h_idx = torch.from_numpy(idx).pin_memory(); h_w = torch.from_numpy(w).pin_memory()
    h_y = torch.empty_like(h_x).pin_memory(); h_dx = torch.empty_like(h_x).pin_memory()
    h_g = [torch.empty(g.shape, dtype=g.dtype).pin_memory() for g in layer.grads]
    slots = [layer, moe.MoELoRALayer(layer.d, layer.w, dev)]
    d_in = [(torch.empty_like(ts["x"]), torch.empty_like(ts["dy"]), torch.empty_like(t_idx), torch.empty_like(t_w))
            for _ in slots]
    bytes_in = sum(t.numel() * t.element_size() for t in (h_x, h_dy, h_idx, h_w))
    bytes_out = sum(t.numel() * t.element_size() for t in (h_y, h_dx, *h_g))
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    computed = [torch.cuda.Event() for _ in slots]     # the slot's step has run
    loaded = [torch.cuda.Event() for _ in slots]       # the slot's inputs are on the device
    fetched = [torch.cuda.Event() for _ in slots]      # the slot's results are on the host

    def e2e_steps(n):
        for i in range(n):
            sl = i % 2
            lay, (d_x, d_dy, d_idx, d_w) = slots[sl], d_in[sl]
            with torch.cuda.stream(up):
                up.wait_event(computed[sl])            # the slot's previous step has read its inputs
                d_x.copy_(h_x, non_blocking=True); d_dy.copy_(h_dy, non_blocking=True)
                d_idx.copy_(h_idx, non_blocking=True); d_w.copy_(h_w, non_blocking=True)
                loaded[sl].record(up)
            stream.wait_event(loaded[sl])
            stream.wait_event(fetched[sl])             # the slot's previous results are out
            lay.step(d_idx, d_w, d_x, d_dy, with_topk_grad=False)
            computed[sl].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(computed[sl])
                h_y.copy_(lay.y, non_blocking=True); h_dx.copy_(lay.dx, non_blocking=True)
                for h, g in zip(h_g, lay.grads):
                    h.copy_(g, non_blocking=True)
                fetched[sl].record(down)

    e2e_steps(4)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(up)
    e2e_steps(args.steps)
    e_end.record(down)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_end), dev)
    clk = clocks.stop()
    e2e_value = job_throughput(cfg.T, args.steps, world, e2e_ms)
    assert all(int(l.dev_status.item()) == 0 for l in slots), "device status flag set"

    # ---- roofline of the dominant kernel and the GEMM aggregate
    peaks = load_peaks()
    work = kernel_work(cfg)
    kernel_ms_step = {n: ms / max(1, args.steps) for n, (ms, cnt) in kt.items()}
    dom = max(kt, key=lambda n: kt[n][0])
    ms_launch = kt[dom][0] / kt[dom][1]
    wk = work[dom]
    t_peak, t_src = tensor_peak(peaks, clk)
    if wk["bound"] == "tensor":
        ach = wk["flops"] / (ms_launch / 1e3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": t_peak,
                "unit": "TFLOP/s", "frac": ach / t_peak,
                "frac_of_sustained": ach / peaks["bf16_tflops_sustained"],
                "traffic": MEASURED_TRAFFIC.get((cfg.name, dom)),
                "algorithmic_flops_per_launch": wk["flops"], "ms_per_launch": ms_launch,
                "sm_mhz_median": clk.get("sm_mhz"), "peak_source": t_src}
    else:
        ach = wk["bytes"] / (ms_launch / 1e3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "traffic": MEASURED_TRAFFIC.get((cfg.name, dom)),
                "algorithmic_bytes_per_launch": wk["bytes"],
                "ms_per_launch": ms_launch, "peak_source": f"{peaks['source']} hbm copy"}
    g_ms = sum(kt[n][0] for n in GEMM_KERNELS if n in kt) / args.steps
    g_fl = sum(work[n]["flops"] for n in GEMM_KERNELS)
    g_tf = g_fl / (g_ms / 1e3) / 1e12 if g_ms > 0 else 0.0
    gemm = {"tflops": g_tf, "frac_of_bf16_peak": g_tf / t_peak, "peak": t_peak, "peak_source": t_src,
            "frac_of_sustained": g_tf / peaks["bf16_tflops_sustained"], "ms_per_step": g_ms, "flops_per_step": g_fl}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(cfg), "clocks": clk,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": bytes_in, "d2h_bytes_per_step": bytes_out},
        "gpu_launches": int(launches),
        "graph_ms_per_step": graph_ms,
        "roofline": roof, "gemm": gemm,
        "layer_tflops": step_flops(cfg) / (total_ms / args.steps / 1e3) / 1e12,
        "wall_s_timed": wall,
        "kernels_ms_per_step": {n: round(v, 4) for n, v in sorted(kernel_ms_step.items(), key=lambda kv: -kv[1])},
        # HBM-bound kernels (routing, gathers, combines, projections, LoRA reductions):
        # algorithmic bytes per launch over the event-timed launch duration
        "kernels_hbm": {n: {"gbs": round(work[n]["bytes"] / (kt[n][0] / kt[n][1] / 1e3) / 1e9, 1),
                            "frac_of_hbm": round(work[n]["bytes"] / (kt[n][0] / kt[n][1] / 1e3) / 1e9
                                                 / peaks["hbm_gbs"], 3)}
                        for n in sorted(kt) if n in work and work[n]["bound"] == "hbm" and kt[n][0] > 0},
        "routing": routing_summary(idx, cfg.E),
    }
    # ---- router step in front of the layer (softmax + top-k and its backward), HBM-bound
    logits = torch.from_numpy(mi.router_logits(cfg, args.seed + rank)).float().to(dev)
    r_idx, r_w = moe.moe_router_topk(logits, cfg.k)
    d_tw = torch.randn((cfg.T, cfg.k), device=dev)
    d_lg = torch.empty_like(logits)
    moe.moe_router_bwd(logits, r_idx, d_tw, d_logits=d_lg)
    torch.cuda.synchronize()
    # device time per launch: each kernel replayed from a CUDA graph of 20 launches (a
    # Python loop of launches would time the host, not these few-microsecond kernels)
    te = cfg.T * cfg.E * 4
    r_bytes = {"router_topk": te + cfg.T * cfg.k * 8, "router_bwd": 2 * te + cfg.T * cfg.k * 8}
    r_ops = {"router_topk": lambda: moe.moe_router_topk(logits, cfg.k, topk_idx=r_idx, topk_w=r_w),
             "router_bwd": lambda: moe.moe_router_bwd(logits, r_idx, d_tw, d_logits=d_lg)}
    # ---- packed-sequence metadata of the batch (samples of up to 2048 tokens: the
    # GPT-OSS-20B-shaped workload's two packed sequences of 2048), built once per batch
    pos = torch.cat([torch.arange(min(2048, cfg.T - b), dtype=torch.int32) for b in range(0, cfg.T, 2048)]).to(dev)
    meta = moe.moe_packed_metadata(pos)
    pmask = moe.moe_packed_causal_mask(meta)
    torch.cuda.synchronize()
    r_bytes["packed_meta"] = cfg.T * 8 + (int(meta.n_seqs.item()) + 1) * 4 + 8
    r_bytes["packed_mask"] = cfg.T * cfg.T + cfg.T * 4
    r_ops["packed_meta"] = lambda: moe.moe_packed_metadata(pos, out=meta)
    r_ops["packed_mask"] = lambda: moe.moe_packed_causal_mask(meta, mask=pmask)
    line["router"] = {}
    gs = torch.cuda.Stream(dev)
    for n, op in r_ops.items():
        gs.wait_stream(stream)
        rg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(rg, stream=gs):
            for _ in range(20):
                op()
        torch.cuda.synchronize()
        reps = max(5, args.steps // 20)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            rg.replay()
        b.record(stream)
        torch.cuda.synchronize()
        us = 1e3 * a.elapsed_time(b) / (20 * reps)
        line["router"][n] = {"us_per_launch": us, "gbs": r_bytes[n] / (us / 1e6) / 1e9}
        del rg
    line["packed_metadata"] = {"T": cfg.T, "n_seqs": int(meta.n_seqs.item()),
                               "max_seqlen": int(meta.max_seqlen.item()),
                               "meta_us": line["router"].pop("packed_meta")["us_per_launch"],
                               **{"mask_" + k: v for k, v in line["router"].pop("packed_mask").items()}}
    # ---- the same step with FP8 (e4m3) and NF4 base weights, dequantised inside the GEMMs
    if not args.no_fp8:
        for fmt in ("fp8", "nf4"):
            line[fmt + "_base"] = quant_measurement(cfg, layer, ts, t_idx, t_w, moe, dev, max(10, args.steps // 4),
                                                    flush, fmt)
    # ---- stack of layers with saved activations offloaded to pinned host memory:
    # backward time with double-buffered reload vs single buffer vs resident
    if not args.no_offload:
        line["offload"] = offload_measurement(cfg, layer, ts, t_idx, t_w, moe, dev, args.offload_layers,
                                              max(3, args.steps // 20))
    # ---- the other workload shapes, a short run each (rank 0 of a single-GPU run)
    if rank == 0 and world == 1 and args.other_steps > 0:
        line["other_configs"] = {}
        for name in ("qwen3_30b", "gptoss120b_skew", "dsv3"):
            if name != cfg.name:
                line["other_configs"][name] = workload_measurement(name, moe, dev, flush, args.other_steps, peaks,
                                                                   args.seed, fp8=not args.no_fp8 and name == "dsv3")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        wts = [ts[n].cpu() for n in ("W_gu", "A_gu", "B_gu", "W_d", "A_d", "B_d")]
        line["cpu_baseline"] = cpu_baseline(cfg, idx, w, ts["x"].cpu(), ts["dy"].cpu(), wts)
    if args.breakdown and rank == 0:
        for n, v in line["kernels_ms_per_step"].items():
            print(f"{n:20s} {v:9.4f} ms/step", file=sys.stderr)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
