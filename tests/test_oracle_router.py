"""Pins for the router part of the oracle (softmax + top-k, its gradient, and the
gradient of the layer w.r.t. the routing weights); no GPU."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as orc


def _f64(t):
    return t.detach().to(torch.float64).numpy()


def test_router_topk_matches_the_workload_recipe():
    for name in ("tiny", "qwen3_30b", "gptoss120b_skew"):
        cfg = mi.CONFIGS[name]
        logits = mi.router_logits(cfg, 0)
        idx, w, p = orc.router_topk(logits, cfg.k)
        ref_idx, ref_w = mi.make_routing(cfg, 0)
        assert np.array_equal(idx, ref_idx)
        np.testing.assert_allclose(w, ref_w, rtol=1e-6)       # recipe stores float32 weights
        np.testing.assert_allclose(p.sum(1), 1.0, rtol=1e-12)


def test_router_topk_ties_and_library_topk():
    z = np.array([[0.5, 2.0, 2.0, -1.0, 2.0], [1.0, 1.0, 1.0, 1.0, 1.0]])
    idx, w, p = orc.router_topk(z, 3)
    assert idx.tolist() == [[1, 2, 4], [0, 1, 2]]
    rng = np.random.default_rng(0)
    z = rng.standard_normal((50, 64))
    idx, w, _ = orc.router_topk(z, 8)
    tv, ti = torch.topk(torch.softmax(torch.tensor(z), dim=1), 8, dim=1)   # distinct values: order unique
    assert np.array_equal(idx, ti.numpy())
    np.testing.assert_allclose(w, tv.numpy(), rtol=1e-12)


def test_router_bwd_against_torch_autograd():
    rng = np.random.default_rng(1)
    z = rng.standard_normal((7, 12))
    idx, w, _ = orc.router_topk(z, 3)
    dw = rng.standard_normal(idx.shape)
    dz = orc.router_bwd(z, idx, dw)
    zt = torch.tensor(z, requires_grad=True)
    wt = torch.gather(torch.softmax(zt, dim=1), 1, torch.tensor(idx))
    (wt * torch.tensor(dw)).sum().backward()
    np.testing.assert_allclose(dz, zt.grad.numpy(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dz.sum(1), 0.0, atol=1e-12)                   # softmax VJP sums to 0


def test_dtopk_w_is_the_exact_directional_derivative():
    cfg = mi.CONFIGS["tiny"]
    idx, w = mi.make_routing(cfg, 0)
    ts = {k: _f64(v) for k, v in mi.make_tensors(cfg, 0, "cpu").items()}
    wts = [ts[n] for n in ("W_gu", "A_gu", "B_gu", "W_d", "A_d", "B_d")]
    dw = orc.lora_dtopk_w(ts["dy"], ts["x"], idx, *wts, cfg.scale)
    L = lambda ww: float((orc.lora_fwd(ts["x"], idx, ww, *wts, cfg.scale) * ts["dy"]).sum())
    w = w.astype(np.float64)
    rng = np.random.default_rng(2)
    for _ in range(12):
        t, j = rng.integers(cfg.T), rng.integers(cfg.k)
        e = np.zeros_like(w); e[t, j] = 1.0
        fd = (L(w + 0.5 * e) - L(w - 0.5 * e))        # y is linear in w: any step is exact
        assert abs(fd - dw[t, j]) <= 1e-10 * max(1.0, abs(dw[t, j]))
    sub = np.array([3, 9])
    dws = orc.lora_dtopk_w(ts["dy"], ts["x"], idx, *wts, cfg.scale, token_subset=sub)
    np.testing.assert_allclose(dws[sub], dw[sub], rtol=1e-12)
    assert np.all(np.delete(dws, sub, axis=0) == 0)


def test_router_and_layer_chain_rule_finite_differences():
    """d L / d logits through top-k (selection held), softmax and the layer, against
    central differences of the composed fp64 function."""
    cfg = mi.micro_config(T=4, E=5, k=2)
    rng = np.random.default_rng(3)
    z = rng.standard_normal((cfg.T, cfg.E)) * 2.0
    ts = {k: _f64(v) * (20.0 if k not in ("x", "dy") else 1.0) for k, v in mi.make_tensors(cfg, 4, "cpu").items()}
    wts = [ts[n] for n in ("W_gu", "A_gu", "B_gu", "W_d", "A_d", "B_d")]
    idx, w, _ = orc.router_topk(z, cfg.k)

    def L(zz):
        ii, ww, _ = orc.router_topk(zz, cfg.k)
        assert np.array_equal(ii, idx), "selection changed under the perturbation"
        return float((orc.lora_fwd(ts["x"], ii, ww, *wts, cfg.scale) * ts["dy"]).sum())

    dz = orc.router_bwd(z, idx, orc.lora_dtopk_w(ts["dy"], ts["x"], idx, *wts, cfg.scale))
    h = 1e-6
    for t in range(cfg.T):
        for e in range(cfg.E):
            zp = z.copy(); zp[t, e] += h
            zm = z.copy(); zm[t, e] -= h
            fd = (L(zp) - L(zm)) / (2 * h)
            assert abs(fd - dz[t, e]) <= 1e-6 * max(1.0, np.abs(dz).max())


def test_mutation_router_bwd_missing_coupling_term_is_caught(monkeypatch):
    def bad(logits, topk_idx, d_topk_w):
        z = np.asarray(logits, np.float64)
        p = np.exp(z - z.max(1, keepdims=True)); p /= p.sum(1, keepdims=True)
        g = np.zeros_like(p); np.put_along_axis(g, np.asarray(topk_idx), np.asarray(d_topk_w), 1)
        return p * g                                           # dropped the "- sum_j dw_j w_j" term
    monkeypatch.setattr(orc, "router_bwd", bad)
    with pytest.raises(AssertionError):
        test_router_bwd_against_torch_autograd()
