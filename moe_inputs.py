"""Seeded synthetic inputs for the MoE-LoRA expert layer.

This module is shared by the CUDA path's tests/bench and by the CPU oracle.
It holds none of the layer's arithmetic: it only draws tensors.  The router
(softmax over E logits, then top-k with ties going to the lower expert index)
is part of the *input recipe* of every workload, not of the layer: the layer
starts from (topk_idx, topk_w).

Workloads (sizes from the MoE-layer shapes of GPT-OSS, Qwen3-MoE and
DeepSeek-V3 that the MoE grouped_mm / Split-LoRA section of the Unsloth 2026
wiki page lists as targets):

  tiny            T=64    H=128  E=8   k=2 I=256  r=8  alpha=16
  gptoss20b       T=4096  H=2880 E=32  k=4 I=2880 r=16 alpha=32
  qwen3_30b       T=8192  H=2048 E=128 k=8 I=768  r=16 alpha=32
  gptoss120b_skew T=16384 H=2880 E=128 k=4 I=2880 r=16 alpha=32 (Zipf-skewed router)
  dsv3            T=4096  H=7168 E=256 k=8 I=2048 r=32 alpha=64

Distributions: x ~ N(0,1); expert W, LoRA A and LoRA B ~ N(0, 0.02) in bf16;
router logits ~ N(0,1) [T,E] (plus 3*log q_e with q_e proportional to
(e+1)^-1.2 for the skewed workload); dY ~ N(0,1).

Tensor layouts (row-major), the same ones the C ABI takes:
  x    [T, H]            W_gu [E, H, 2I]  (gate = cols [0,I), up = cols [I,2I))
  W_d  [E, I, H]         A_gu [E, r, H]   (LoRA A stored transposed, r x in)
  B_gu [E, r, 2I]        A_d  [E, r, I]   B_d [E, r, H]
  topk_idx [T, k] int64, topk_w [T, k] float32, dy [T, H]
"""
from __future__ import annotations

import dataclasses
import hashlib

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    r: int
    alpha: float
    zipf_s: float = 0.0      # > 0: add 3*log(Zipf(s) rank weight) to expert logits
    w_std: float = 0.02

    @property
    def scale(self) -> float:
        """LoRA scale s = alpha / r (the usual PEFT convention; the pages do not fix it)."""
        return float(self.alpha) / float(self.r)

    @property
    def N(self) -> int:
        return self.T * self.k

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny": MoEConfig("tiny", T=64, H=128, E=8, k=2, I=256, r=8, alpha=16),
    "gptoss20b": MoEConfig("gptoss20b", T=4096, H=2880, E=32, k=4, I=2880, r=16, alpha=32),
    "qwen3_30b": MoEConfig("qwen3_30b", T=8192, H=2048, E=128, k=8, I=768, r=16, alpha=32),
    "gptoss120b_skew": MoEConfig("gptoss120b_skew", T=16384, H=2880, E=128, k=4, I=2880,
                                 r=16, alpha=32, zipf_s=1.2),
    "dsv3": MoEConfig("dsv3", T=4096, H=7168, E=256, k=8, I=2048, r=32, alpha=64),
}

TENSOR_NAMES = ("x", "W_gu", "A_gu", "B_gu", "W_d", "A_d", "B_d", "dy")


def _sub_seed(seed: int, name: str) -> int:
    h = hashlib.sha256(f"{seed}:{name}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 62) - 1)


def tensor_shape(cfg: MoEConfig, name: str) -> tuple:
    T, H, E, I, r = cfg.T, cfg.H, cfg.E, cfg.I, cfg.r
    return {
        "x": (T, H), "dy": (T, H),
        "W_gu": (E, H, 2 * I), "W_d": (E, I, H),
        "A_gu": (E, r, H), "B_gu": (E, r, 2 * I),
        "A_d": (E, r, I), "B_d": (E, r, H),
    }[name]


def tensor_std(cfg: MoEConfig, name: str) -> float:
    return 1.0 if name in ("x", "dy") else cfg.w_std


def make_tensor(cfg: MoEConfig, name: str, seed: int = 0, device="cpu",
                dtype=torch.bfloat16) -> torch.Tensor:
    """One named input tensor, drawn from its own generator (independent of draw order).

    The values depend on the device's generator (CPU and CUDA draw different streams);
    a workload is defined by (config, seed, device)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(_sub_seed(seed, name))
    shape = tensor_shape(cfg, name)
    std = tensor_std(cfg, name)
    t = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def make_tensors(cfg: MoEConfig, seed: int = 0, device="cpu", names=TENSOR_NAMES) -> dict:
    return {n: make_tensor(cfg, n, seed, device) for n in names}


def router_logits(cfg: MoEConfig, seed: int = 0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(_sub_seed(seed, "router")))
    logits = rng.standard_normal((cfg.T, cfg.E))
    if cfg.zipf_s > 0:
        q = (np.arange(1, cfg.E + 1, dtype=np.float64)) ** (-cfg.zipf_s)
        q /= q.sum()
        logits = logits + 3.0 * np.log(q)[None, :]
    return logits


def make_routing(cfg: MoEConfig, seed: int = 0):
    """Router input recipe: softmax over all E logits (fp64), then the k largest
    probabilities in descending order, ties to the lower expert index; no
    renormalisation.  Returns topk_idx [T,k] int64 and topk_w [T,k] float32."""
    logits = router_logits(cfg, seed)
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    # stable argsort of -p: equal probabilities keep ascending expert order
    order = np.argsort(-p, axis=1, kind="stable")[:, : cfg.k]
    topk_idx = order.astype(np.int64)
    topk_w = np.take_along_axis(p, order, axis=1).astype(np.float32)
    return topk_idx, topk_w


def micro_config(**kw) -> MoEConfig:
    """A very small layer for finite differences and brute force."""
    base = dict(name="micro", T=6, H=8, E=3, k=2, I=8, r=2, alpha=4)
    base.update(kw)
    return MoEConfig(**base)
