"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: a library
routine, brute force, an independently written formula (per-token split-LoRA
instead of per-expert merged), autograd, finite differences, a hand-worked
case, or a special case with a textbook answer.  The mutation tests at the end
plant a plausible mistake in the oracle and check that a pin catches it.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import moe_inputs as mi
from oracle import moe_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f64(t):
    return t.detach().to(torch.float64).numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def _layer(cfg, seed=0, zero_B=False):
    idx, w = mi.make_routing(cfg, seed)
    ts = mi.make_tensors(cfg, seed, "cpu")
    ts = {k: _f64(v) for k, v in ts.items()}
    if zero_B:
        ts["B_gu"][:] = 0.0
        ts["B_d"][:] = 0.0
    return idx, w.astype(np.float64), ts


def _fwd(cfg, idx, w, ts, **kw):
    return orc.lora_fwd(ts["x"], idx, w, ts["W_gu"], ts["A_gu"], ts["B_gu"], ts["W_d"],
                        ts["A_d"], ts["B_d"], cfg.scale, **kw)


def _bwd(cfg, idx, w, ts, **kw):
    return orc.lora_bwd(ts["dy"], ts["x"], idx, w, ts["W_gu"], ts["A_gu"], ts["B_gu"],
                        ts["W_d"], ts["A_d"], ts["B_d"], cfg.scale, **kw)


# ---------------------------------------------------------------- routing
ROUTE_CASES = [("tiny", 0), ("tiny", 1), ("qwen3_30b", 0), ("gptoss120b_skew", 0)]


@pytest.mark.parametrize("name,seed", ROUTE_CASES)
def test_route_invariants(name, seed):
    cfg = mi.CONFIGS[name]
    idx, _ = mi.make_routing(cfg, seed)
    counts, offsets, perm, inv_perm = orc.route(idx, cfg.E)
    flat = idx.reshape(-1)
    N = cfg.T * cfg.k
    assert counts.sum() == N
    assert offsets[0] == 0 and offsets[-1] == N and np.all(np.diff(offsets) == counts)
    assert np.array_equal(np.sort(perm), np.arange(N))             # bijection
    for e in range(cfg.E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)                            # stable: ascending flat index
    assert np.array_equal(inv_perm[perm], np.arange(N))


@pytest.mark.parametrize("name,seed", ROUTE_CASES)
def test_route_matches_library_stable_sort(name, seed):
    cfg = mi.CONFIGS[name]
    idx, _ = mi.make_routing(cfg, seed)
    counts, offsets, perm, _ = orc.route(idx, cfg.E)
    flat = idx.reshape(-1)
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))
    assert np.array_equal(counts, np.bincount(flat, minlength=cfg.E))


def test_route_bruteforce_all_assignments():
    # every assignment of T*k slots to E experts, T <= 3, k <= 2, E <= 3
    for T, k, E in [(1, 1, 1), (2, 1, 3), (3, 1, 2), (2, 2, 3), (3, 2, 3)]:
        for flat in itertools.product(range(E), repeat=T * k):
            idx = np.array(flat, dtype=np.int64).reshape(T, k)
            counts, offsets, perm, inv = orc.route(idx, E)
            expect = sorted(range(T * k), key=lambda i: (flat[i], i))
            assert perm.tolist() == expect
            assert counts.tolist() == [flat.count(e) for e in range(E)]


def test_route_empty_experts_and_skew():
    cfg = mi.CONFIGS["gptoss120b_skew"]
    idx, _ = mi.make_routing(cfg, 0)
    counts, _, _, _ = orc.route(idx, cfg.E)
    mean = cfg.T * cfg.k / cfg.E
    assert (counts == 0).sum() >= 10, "skewed router should leave many experts empty"
    assert counts.max() > 10 * mean, "skewed router should overload a few experts"


def test_route_rejects_out_of_range():
    with pytest.raises(ValueError):
        orc.route(np.array([[0, 3]]), 3)


def test_tile_offsets():
    t = orc.tile_offsets(np.array([0, 1, 128, 129, 256]), 128)
    assert t.tolist() == [0, 0, 1, 2, 4, 6]


def test_routing_recipe_ties_go_to_lower_expert():
    # equal logits for every expert: top-k must be experts 0..k-1 in order
    cfg = mi.micro_config(T=2, E=5, k=3)
    logits = np.zeros((cfg.T, cfg.E))
    z = np.exp(logits - logits.max(1, keepdims=True)); p = z / z.sum(1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :cfg.k]
    assert order.tolist() == [[0, 1, 2], [0, 1, 2]]
    idx, w = mi.make_routing(cfg, 0)
    assert np.all(np.diff(w, axis=1) <= 0)                         # descending weights
    assert all(len(set(row)) == cfg.k for row in idx.tolist())     # no duplicates


# ---------------------------------------------------------------- golden hand-worked cases
def test_golden_route_hand_case():
    with open(os.path.join(GOLDEN, "route_hand_case.json")) as f:
        case = json.load(f)
    counts, offsets, perm, inv = orc.route(np.array(case["topk_idx"]), case["E"])
    assert counts.tolist() == case["counts"]
    assert offsets.tolist() == case["offsets"]
    assert perm.tolist() == case["perm"]
    assert inv.tolist() == case["inv_perm"]


def test_golden_layer_hand_case():
    with open(os.path.join(GOLDEN, "layer_hand_case.json")) as f:
        c = json.load(f)
    def ev(v):
        if isinstance(v, list):
            return [ev(u) for u in v]
        return eval(v, {"log": np.log}) if isinstance(v, str) else v

    a = lambda k: np.array(ev(c["inputs"][k]), dtype=np.float64)
    y = orc.lora_fwd(a("x"), np.array(c["inputs"]["topk_idx"]), a("topk_w"), a("W_gu"), a("A_gu"),
                     a("B_gu"), a("W_d"), a("A_d"), a("B_d"), c["inputs"]["scale"])
    expect = eval(c["expected_y_expr"], {"log": np.log})  # closed form written in the fixture
    np.testing.assert_allclose(y.reshape(-1), np.array(expect, dtype=np.float64).reshape(-1),
                               rtol=1e-13, atol=1e-15)
    dx, dA_gu, dB_gu, dA_d, dB_d = orc.lora_bwd(
        a("dy"), a("x"), np.array(c["inputs"]["topk_idx"]), a("topk_w"), a("W_gu"), a("A_gu"),
        a("B_gu"), a("W_d"), a("A_d"), a("B_d"), c["inputs"]["scale"])
    for name, got in (("dx", dx), ("dA_d", dA_d), ("dB_d", dB_d)):
        want = np.array(eval(c["expected_grad_exprs"][name], {"log": np.log}), dtype=np.float64)
        np.testing.assert_allclose(got.reshape(-1), want.reshape(-1), rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- forward pins
def _split_per_token(cfg, idx, w, ts):
    """Split-LoRA written per token and per slot: x W + s (x A) B, never merged."""
    T, H = ts["x"].shape
    I = cfg.I
    y = np.zeros((T, H))
    for t in range(T):
        for j in range(cfg.k):
            e = idx[t, j]
            xt = ts["x"][t]
            gu = xt @ ts["W_gu"][e] + cfg.scale * ((ts["A_gu"][e] @ xt) @ ts["B_gu"][e])
            g, u = gu[:I], gu[I:]
            h = g * expit(g) * u
            o = h @ ts["W_d"][e] + cfg.scale * ((ts["A_d"][e] @ h) @ ts["B_d"][e])
            y[t] += w[t, j] * o
    return y


@pytest.mark.parametrize("cfg", [mi.micro_config(), mi.CONFIGS["tiny"]], ids=["micro", "tiny"])
def test_split_lora_equals_merged(cfg):
    idx, w, ts = _layer(cfg)
    y = _fwd(cfg, idx, w, ts)
    y2 = _split_per_token(cfg, idx, w, ts)
    np.testing.assert_allclose(y, y2, rtol=1e-11, atol=1e-12 * np.abs(y2).max())


def test_B_zero_gives_base_layer_and_zero_dA():
    cfg = mi.CONFIGS["tiny"]
    idx, w, ts = _layer(cfg, zero_B=True)
    y = _fwd(cfg, idx, w, ts)
    base = {**ts, "A_gu": np.zeros_like(ts["A_gu"]), "A_d": np.zeros_like(ts["A_d"])}
    np.testing.assert_allclose(y, _split_per_token(cfg, idx, w, base), rtol=1e-11, atol=1e-13)
    dx, dA_gu, dB_gu, dA_d, dB_d = _bwd(cfg, idx, w, ts)
    assert np.all(dA_gu == 0.0) and np.all(dA_d == 0.0)           # exactly zero
    assert np.abs(dB_gu).max() > 0 and np.abs(dB_d).max() > 0


def test_E1_k1_is_dense_swiglu_mlp_torch_autograd():
    """E = 1, k = 1: the softmax weight is 1 and the layer is a dense SwiGLU MLP with
    weights W + s A B.  Compare y and all gradients with torch fp64 + autograd."""
    cfg = mi.micro_config(T=5, H=12, E=1, k=1, I=10, r=3, alpha=6)
    idx, w, ts = _layer(cfg, seed=3)
    assert np.all(idx == 0) and np.allclose(w, 1.0)
    y = _fwd(cfg, idx, w, ts)
    grads = _bwd(cfg, idx, w, ts)

    tt = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in ts.items()}
    F = torch.nn.functional
    Wg = tt["W_gu"][0] + cfg.scale * tt["A_gu"][0].T @ tt["B_gu"][0]
    Wd = tt["W_d"][0] + cfg.scale * tt["A_d"][0].T @ tt["B_d"][0]
    gu = F.linear(tt["x"], Wg.T)
    h = F.silu(gu[:, :cfg.I]) * gu[:, cfg.I:]
    yt = F.linear(h, Wd.T) * torch.tensor(w, dtype=torch.float64)
    np.testing.assert_allclose(y, yt.detach().numpy(), rtol=1e-12, atol=1e-14)
    (yt * tt["dy"]).sum().backward()
    for got, name in zip(grads, ["x", "A_gu", "B_gu", "A_d", "B_d"]):
        np.testing.assert_allclose(got, tt[name].grad.numpy(), rtol=1e-10, atol=1e-13)


def test_token_permutation_equivariance_and_linearity_in_w():
    cfg = mi.CONFIGS["tiny"]
    idx, w, ts = _layer(cfg, seed=2)
    y = _fwd(cfg, idx, w, ts)
    rng = np.random.default_rng(0)
    pi = rng.permutation(cfg.T)
    ts2 = dict(ts, x=ts["x"][pi], dy=ts["dy"][pi])
    y2 = _fwd(cfg, idx[pi], w[pi], ts2)
    np.testing.assert_allclose(y2, y[pi], rtol=1e-12, atol=1e-14)
    dx = _bwd(cfg, idx, w, ts)[0]
    dx2 = _bwd(cfg, idx[pi], w[pi], ts2)[0]
    np.testing.assert_allclose(dx2, dx[pi], rtol=1e-12, atol=1e-14)
    y3 = _fwd(cfg, idx, 2.5 * w, ts)
    np.testing.assert_allclose(y3, 2.5 * y, rtol=1e-12, atol=1e-14)


def test_token_and_expert_subsets_match_full():
    cfg = mi.CONFIGS["tiny"]
    idx, w, ts = _layer(cfg, seed=1)
    sub = np.array([0, 5, 17, 63])
    y = _fwd(cfg, idx, w, ts)
    ys = _fwd(cfg, idx, w, ts, token_subset=sub)
    np.testing.assert_allclose(ys[sub], y[sub], rtol=1e-12, atol=1e-15)
    assert np.all(np.delete(ys, sub, axis=0) == 0)
    full = _bwd(cfg, idx, w, ts)
    part = _bwd(cfg, idx, w, ts, token_subset=sub, expert_subset=[1, 6])
    np.testing.assert_allclose(part[0][sub], full[0][sub], rtol=1e-12, atol=1e-14)
    for g_full, g_part in zip(full[1:], part[1:]):
        np.testing.assert_allclose(g_part[[1, 6]], g_full[[1, 6]], rtol=1e-12, atol=1e-14)
        assert np.all(g_part[[0, 2, 3, 4, 5, 7]] == 0)


# ---------------------------------------------------------------- gradient pins
def _loss(cfg, idx, w, ts):
    return float((_fwd(cfg, idx, w, ts) * ts["dy"]).sum())


def _fd_check(cfg, idx, w, ts, names, max_entries=None, seed=0, h=1e-6, rtol=1e-6):
    grads = dict(zip(["x", "A_gu", "B_gu", "A_d", "B_d"], _bwd(cfg, idx, w, ts)))
    rng = np.random.default_rng(seed)
    for name in names:
        g = grads[name]
        flat_n = g.size
        picks = np.arange(flat_n) if max_entries is None else rng.choice(flat_n, max_entries, replace=False)
        for f in picks:
            ii = np.unravel_index(f, g.shape)
            p = {k: v.copy() for k, v in ts.items()}
            p[name][ii] += h
            lp = _loss(cfg, idx, w, p)
            p[name][ii] -= 2 * h
            lm = _loss(cfg, idx, w, p)
            fd = (lp - lm) / (2 * h)
            scale = max(np.abs(g).max(), 1e-30)
            assert abs(fd - g[ii]) <= rtol * scale + 1e-9, (name, ii, fd, g[ii])


def test_finite_differences_micro_full_jacobian():
    cfg = mi.micro_config()
    idx, w, ts = _layer(cfg, seed=5)
    # scale weights up so the nonlinearity is exercised
    for k in ("W_gu", "W_d", "A_gu", "B_gu", "A_d", "B_d"):
        ts[k] = ts[k] * 20.0
    _fd_check(cfg, idx, w, ts, ["x", "A_gu", "B_gu", "A_d", "B_d"])


def test_finite_differences_tiny_sampled():
    cfg = mi.CONFIGS["tiny"]
    idx, w, ts = _layer(cfg, seed=0)
    _fd_check(cfg, idx, w, ts, ["x", "A_gu", "B_gu", "A_d", "B_d"], max_entries=12)


def test_swiglu_bwd_scalar_fd():
    rng = np.random.default_rng(1)
    for _ in range(50):
        g, u, dh = rng.standard_normal(3) * 3
        gu = np.array([[g, u]])
        d = orc.swiglu_bwd(np.array([[dh]]), gu, 1)[0]
        h = 1e-6
        f = lambda gg, uu: dh * orc.swiglu(np.array([[gg, uu]]), 1)[0, 0]
        assert abs(d[0] - (f(g + h, u) - f(g - h, u)) / (2 * h)) < 1e-7 * (1 + abs(d[0]))
        assert abs(d[1] - (f(g, u + h) - f(g, u - h)) / (2 * h)) < 1e-7 * (1 + abs(d[1]))


def test_silu_matches_torch():
    z = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(orc.silu(z), torch.nn.functional.silu(torch.tensor(z)).numpy(),
                               rtol=1e-14, atol=1e-300)


# ---------------------------------------------------------------- mutation tests
def _mutant_checks(monkeypatch, attr, bad):
    """Plant `bad` in place of oracle.`attr` and return which pins still pass."""
    monkeypatch.setattr(orc, attr, bad)
    cfg = mi.micro_config()
    idx, w, ts = _layer(cfg, seed=5)
    for k in ("W_gu", "W_d", "A_gu", "B_gu", "A_d", "B_d"):
        ts[k] = ts[k] * 20.0
    fwd_ok = np.allclose(_fwd(cfg, idx, w, ts), _split_per_token(cfg, idx, w, ts), rtol=1e-9)
    try:
        _fd_check(cfg, idx, w, ts, ["x", "A_gu", "B_gu", "A_d", "B_d"], max_entries=10)
        bwd_ok = True
    except AssertionError:
        bwd_ok = False
    return fwd_ok, bwd_ok


def test_mutation_swapped_gate_up_is_caught(monkeypatch):
    orig = orc.swiglu
    fwd_ok, _ = _mutant_checks(monkeypatch, "swiglu",
                               lambda gu, I: orig(np.concatenate([gu[:, I:], gu[:, :I]], 1), I))
    assert not fwd_ok


def test_mutation_dropped_lora_term_is_caught(monkeypatch):
    fwd_ok, _ = _mutant_checks(monkeypatch, "merged", lambda W, A, B, s: W)
    assert not fwd_ok


def test_mutation_swiglu_bwd_sign_is_caught(monkeypatch):
    def bad(dh, gu, I):
        g, u = gu[:, :I], gu[:, I:]
        sg = orc.sigmoid(g)
        return np.concatenate([dh * u * sg * (1.0 - g * (1.0 - sg)), dh * g * sg], 1)
    fwd_ok, bwd_ok = _mutant_checks(monkeypatch, "swiglu_bwd", bad)
    assert fwd_ok and not bwd_ok
