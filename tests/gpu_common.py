"""Helpers shared by the GPU parity tests (inputs on the device, oracle on CPU)."""
from __future__ import annotations

import numpy as np
import torch

import moe_inputs as mi

REL_L2 = 5e-3        # relative L2 error bound for bf16 outputs and gradients
MAX_ABS = 2e-2       # max-abs error bound, relative to max |oracle|
WEIGHT_NAMES = ("W_gu", "A_gu", "B_gu", "W_d", "A_d", "B_d")


class LazyExperts:
    """Per-expert host view of a device expert stack: the oracle reads W[e] one
    expert at a time, so only the experts it touches are copied to the host."""

    def __init__(self, t: torch.Tensor):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, e):
        return self.t[e].to("cpu")


def make_case(cfg: mi.MoEConfig, seed: int = 0, device="cuda", gen_device=None, zero_B=False):
    """Seeded inputs for `cfg` on the device.  Small layers are drawn on the CPU
    generator and copied; large ones on the CUDA generator."""
    if gen_device is None:
        gen_device = "cpu" if 3 * cfg.E * cfg.H * cfg.I <= 50_000_000 else device
    idx, w = mi.make_routing(cfg, seed)
    ts = mi.make_tensors(cfg, seed, gen_device)
    ts = {k: v.to(device) for k, v in ts.items()}
    if zero_B:
        ts["B_gu"].zero_()
        ts["B_d"].zero_()
    return idx, w, ts


def run_layer(cfg, idx, w, ts, idx_dtype=torch.int64, with_topk_grad=True, h_from_gu=False):
    import moe_expert_dispatch_stable_gb300 as moe
    dev = ts["x"].device
    d = moe.Dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r, cfg.scale)
    layer = moe.MoELoRALayer(d, ts, dev, h_from_gu=h_from_gu)
    grads = layer.step(torch.from_numpy(idx).to(dev, idx_dtype), torch.from_numpy(w).to(dev), ts["x"], ts["dy"],
                       with_topk_grad=with_topk_grad)
    torch.cuda.synchronize()
    return layer, grads


def to64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def errors(got: np.ndarray, ref: np.ndarray):
    den = max(np.linalg.norm(ref), 1e-30)
    rel = float(np.linalg.norm(got - ref) / den)
    mx = float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30)) if ref.size else 0.0
    return rel, mx


def assert_elementwise(name: str, got: np.ndarray, ref: np.ndarray):
    """The per-element half of the bound alone: |got - ref| <= 2e-2 * max|ref| everywhere."""
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    if ref.size == 0:
        return
    if np.abs(ref).max() == 0:
        assert np.abs(got).max() == 0, f"{name}: expected exact zeros"
        return
    _, mx = errors(got, ref)
    assert mx <= MAX_ABS, f"{name}: max-abs/max {mx:.3e} (<= {MAX_ABS})"


def assert_close(name: str, got: np.ndarray, ref: np.ndarray):
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    if ref.size == 0:
        return
    if np.abs(ref).max() == 0:
        assert np.abs(got).max() == 0, f"{name}: expected exact zeros"
        return
    rel, mx = errors(got, ref)
    assert rel <= REL_L2 and mx <= MAX_ABS, f"{name}: rel-L2 {rel:.3e} (<= {REL_L2}), max-abs/max {mx:.3e} (<= {MAX_ABS})"
