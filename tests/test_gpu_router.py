"""GPU parity of the router step (softmax + top-k and its backward) and of the
routing-weight gradient of the layer, against the CPU oracle."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as orc
from tests.gpu_common import (WEIGHT_NAMES, LazyExperts, assert_close, errors, make_case, run_layer, to64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("name", list(mi.CONFIGS))
def test_router_topk_indices_bit_exact_weights_close(name):
    import moe_expert_dispatch_stable_gb300 as moe
    cfg = mi.CONFIGS[name]
    for seed in (0, 1):
        logits = torch.from_numpy(mi.router_logits(cfg, seed)).float()
        idx, w = moe.moe_router_topk(logits.cuda(), cfg.k)
        torch.cuda.synchronize()
        ref_idx, ref_w, _ = orc.router_topk(logits.numpy(), cfg.k)
        assert np.array_equal(idx.cpu().numpy(), ref_idx)
        np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=2e-6, atol=1e-9)


def test_router_topk_ties_go_to_lower_index():
    import moe_expert_dispatch_stable_gb300 as moe
    z = torch.tensor([[0.5, 2.0, 2.0, -1.0, 2.0], [1.0, 1.0, 1.0, 1.0, 1.0], [-3.0, 0.0, -3.0, 0.0, 0.0]])
    idx, w = moe.moe_router_topk(z.cuda(), 3)
    torch.cuda.synchronize()
    assert idx.cpu().tolist() == [[1, 2, 4], [0, 1, 2], [1, 3, 4]]
    # E = k (every expert selected) and E = 1024
    for T, E, k in [(5, 7, 7), (33, 1024, 8)]:
        z = torch.randn(T, E)
        idx, w = moe.moe_router_topk(z.cuda(), k)
        ref_idx, ref_w, _ = orc.router_topk(z.numpy(), k)
        assert np.array_equal(idx.cpu().numpy(), ref_idx)
        np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=2e-6, atol=1e-9)


@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (4096, 32, 4), (300, 256, 8), (17, 1024, 3)])
def test_router_bwd_matches_oracle(T, E, k):
    import moe_expert_dispatch_stable_gb300 as moe
    g = torch.Generator().manual_seed(T + E)
    z = torch.randn(T, E, generator=g) * 2
    idx, _, _ = orc.router_topk(z.numpy(), k)
    dw = torch.randn(T, k, generator=g)
    dz = moe.moe_router_bwd(z.cuda(), torch.from_numpy(idx).int().cuda(), dw.cuda())
    torch.cuda.synchronize()
    ref = orc.router_bwd(z.numpy(), idx, dw.numpy())
    rel, mx = errors(dz.double().cpu().numpy(), ref)
    assert rel <= 1e-5 and mx <= 1e-5, (rel, mx)


@pytest.mark.parametrize("name", ["tiny", "skew_small"])
def test_d_topk_w_matches_oracle(name):
    from tests.test_gpu_parity import SMALL_CASES
    cfg = SMALL_CASES[name]
    idx, w, ts = make_case(cfg, seed=0)
    layer, _ = run_layer(cfg, idx, w, ts)
    c = {k: v.cpu() for k, v in ts.items()}
    ref = orc.lora_dtopk_w(c["dy"], c["x"], idx, *[c[n] for n in WEIGHT_NAMES], cfg.scale)
    assert_close("d_topk_w", to64(layer.d_topk_w), ref)


def test_router_to_d_logits_chain():
    """logits -> router (GPU) -> route -> forward -> backward with d_topk_w -> router
    backward (GPU), against the oracle's composition of the same steps."""
    import moe_expert_dispatch_stable_gb300 as moe
    from tests.test_gpu_parity import SMALL_CASES
    cfg = SMALL_CASES["ragged"]
    _, _, ts = make_case(cfg, seed=5)
    logits = torch.from_numpy(mi.router_logits(cfg, 5)).float()
    lz = logits.cuda()
    idx, w = moe.moe_router_topk(lz, cfg.k)
    d = moe.Dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r, cfg.scale)
    layer = moe.MoELoRALayer(d, ts)
    layer.step(idx, w, ts["x"], ts["dy"])
    dz = moe.moe_router_bwd(lz, idx, layer.d_topk_w)
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    ref_idx, ref_w, _ = orc.router_topk(logits.numpy(), cfg.k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    c = {k: v.cpu() for k, v in ts.items()}
    wts = [c[n] for n in WEIGHT_NAMES]
    assert_close("y", to64(layer.y), orc.lora_fwd(c["x"], ref_idx, ref_w, *wts, cfg.scale))
    dw_ref = orc.lora_dtopk_w(c["dy"], c["x"], ref_idx, *wts, cfg.scale)
    assert_close("d_topk_w", to64(layer.d_topk_w), dw_ref)
    assert_close("d_logits", dz.double().cpu().numpy(), orc.router_bwd(logits.numpy(), ref_idx, dw_ref))


@pytest.mark.parametrize("name", ["gptoss20b", "dsv3"])
def test_d_topk_w_full_size_sampled(name):
    cfg = mi.CONFIGS[name]
    idx, w, ts = make_case(cfg, seed=0)
    layer, _ = run_layer(cfg, idx, w, ts)
    toks = np.sort(np.random.default_rng(1).choice(cfg.T, 12, replace=False))
    lazy = [LazyExperts(ts[n]) for n in WEIGHT_NAMES]
    ref = orc.lora_dtopk_w(ts["dy"].cpu(), ts["x"].cpu(), idx, *lazy, cfg.scale, token_subset=toks)
    assert_close("d_topk_w[sample]", to64(layer.d_topk_w)[toks], ref[toks])
