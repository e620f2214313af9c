"""A stack of MoE-LoRA layers whose saved activations live in pinned host memory
between forward and backward gives bit-identical results to the same stack with
every layer's activations kept on the device (same kernels, same inputs)."""
import pytest
import torch

import moe_inputs as mi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _stack_inputs(cfg, L):
    weights, routing = [], []
    for l in range(L):
        ts = mi.make_tensors(cfg, 10 + l, "cpu", names=("W_gu", "A_gu", "B_gu", "W_d", "A_d", "B_d"))
        weights.append({k: v.cuda() for k, v in ts.items()})
        idx, w = mi.make_routing(cfg, 10 + l)
        routing.append((torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()))
    x0 = mi.make_tensor(cfg, "x", 0, "cpu").cuda()
    dy = mi.make_tensor(cfg, "dy", 0, "cpu").cuda()
    return weights, routing, x0, dy


@pytest.mark.parametrize("buffers", [2, 1, "auto"])
@pytest.mark.parametrize("L", [1, 3])
def test_offloaded_stack_is_bit_identical_to_resident(buffers, L):
    import moe_expert_dispatch_stable_gb300 as moe
    from moe_expert_dispatch_stable_gb300.offload import OffloadedMoEStack
    cfg = mi.MoEConfig("stack", T=700, H=256, E=6, k=2, I=320, r=16, alpha=32)
    d = moe.Dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r, cfg.scale)
    weights, routing, x0, dy = _stack_inputs(cfg, L)

    layers = [moe.MoELoRALayer(d, w, h_from_gu=True) for w in weights]   # the stack's forward
    x = x0
    for l in range(L):
        layers[l].route(*routing[l])
        x = layers[l].forward(x)
    g = dy
    for l in range(L - 1, -1, -1):
        g = layers[l].backward(g, with_topk_grad=False)[0]
    torch.cuda.synchronize()

    stack = OffloadedMoEStack(d, weights, buffers=buffers)
    y = stack.forward(x0, routing)
    dx0 = stack.backward(dy)
    torch.cuda.synchronize()
    assert int(stack.dev_status.item()) == 0
    assert torch.equal(y, layers[-1].y)
    assert torch.equal(dx0, layers[0].dx)
    for l in range(L):
        for a, b in zip(stack.grads[l], layers[l].grads):
            assert torch.equal(a, b)
    # a second pass over the same buffers gives the same answer again
    y2 = stack.forward(x0, routing).clone()
    dx2 = stack.backward(dy).clone()
    torch.cuda.synchronize()
    assert torch.equal(y2, y) and torch.equal(dx2, dx0)


def test_saved_regather_reproduces_x_perm_bit_for_bit():
    import moe_expert_dispatch_stable_gb300 as moe
    cfg = mi.MoEConfig("regather", T=300, H=128, E=5, k=2, I=192, r=8, alpha=16)
    d = moe.Dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r, cfg.scale)
    weights, routing, x0, _ = _stack_inputs(cfg, 1)
    layer = moe.MoELoRALayer(d, weights[0])
    layer.route(*routing[0])
    layer.forward(x0)
    offs, _ = moe.moe_lora_saved_layout(d)
    N = cfg.T * cfg.k
    ref = layer.saved.clone()
    layer.saved[offs[0]:offs[0] + N * cfg.H * 2].fill_(0x5A)      # scribble over the x_perm rows only
    moe.moe_lora_saved_regather(d, layer.rt, x0, layer.saved)
    torch.cuda.synchronize()
    assert torch.equal(layer.saved, ref)
    # the section really is x gathered in expert order
    xp = layer.saved[offs[0]:offs[0] + N * cfg.H * 2].view(torch.bfloat16).view(N, cfg.H)
    perm = layer.rt.perm.long()
    assert torch.equal(xp, x0[perm // cfg.k])


@pytest.mark.parametrize("name", ["small", "pairs", "gptoss20b"])
def test_saved_rebuild_h_reproduces_h_bit_for_bit(name):
    """moe_lora_fwd_h_from_gu forms h from the bf16 GU it stores; moe_lora_saved_rebuild_h
    recomputes h from that GU alone, bit for bit (single-CTA and SM-pair tiles, and the
    GPT-OSS-20B shape in full), and touches nothing else in `saved`."""
    import moe_expert_dispatch_stable_gb300 as moe
    cfg = {"small": mi.MoEConfig("regather", T=300, H=128, E=5, k=2, I=192, r=8, alpha=16),
           "pairs": mi.MoEConfig("pairs", T=1000, H=256, E=4, k=2, I=320, r=16, alpha=32),
           "gptoss20b": mi.CONFIGS["gptoss20b"]}[name]
    d = moe.Dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r, cfg.scale)
    weights, routing, x0, _ = _stack_inputs(cfg, 1)
    layer = moe.MoELoRALayer(d, weights[0], h_from_gu=True)
    layer.route(*routing[0])
    layer.forward(x0)
    offs, _ = moe.moe_lora_saved_layout(d)
    N = cfg.T * cfg.k
    ref = layer.saved.clone()
    layer.saved[offs[2]:offs[2] + N * cfg.I * 2].fill_(0x5A)      # scribble over the h rows only
    moe.moe_lora_saved_rebuild_h(d, layer.saved)
    torch.cuda.synchronize()
    assert torch.equal(layer.saved, ref)


def test_offloaded_stack_matches_oracle():
    """A 3-layer stack with double-buffered reload of its offloaded activations against
    the fp64 oracle, layer by layer: layer l's y, its dx and its four LoRA gradients.
    The oracle of layer l takes the stack's own bf16 input of that layer (x_0, then
    y_{l-1}) and, in the backward, the bf16 gradient the stack passed into it (dy, then
    dx_{l+1}), so the bound applies to each layer on its own and does not compound."""
    import numpy as np
    from moe_expert_dispatch_stable_gb300.offload import OffloadedMoEStack
    import moe_expert_dispatch_stable_gb300 as moe
    from oracle import moe_oracle as orc
    from tests.gpu_common import WEIGHT_NAMES, assert_close, to64
    L = 3
    cfg = mi.MoEConfig("stack", T=700, H=256, E=6, k=2, I=320, r=16, alpha=32)
    d = moe.Dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r, cfg.scale)
    weights, routing, x0, dy = _stack_inputs(cfg, L)
    stack = OffloadedMoEStack(d, weights, buffers=2)
    assert stack.n_buf == 2
    stack.forward(x0, routing)
    stack.backward(dy)
    torch.cuda.synchronize()
    assert int(stack.dev_status.item()) == 0
    for l in range(L):
        x_in = (x0 if l == 0 else stack.y[l - 1]).cpu()
        g_in = (dy if l == L - 1 else stack.dx[l + 1]).cpu()
        idx, w = routing[l][0].cpu().numpy(), routing[l][1].cpu().numpy()
        wts = [weights[l][n].cpu() for n in WEIGHT_NAMES]
        y_ref = orc.lora_fwd(x_in, idx, w, *wts, cfg.scale)
        assert_close(f"y[{l}]", to64(stack.y[l]), y_ref)
        g_ref = orc.lora_bwd(g_in, x_in, idx, w, *wts, cfg.scale)
        assert_close(f"dx[{l}]", to64(stack.dx[l]), g_ref[0])
        for nm, got, ref in zip(["dA_gu", "dB_gu", "dA_d", "dB_d"], stack.grads[l], g_ref[1:]):
            assert_close(f"{nm}[{l}]", to64(got), ref)
        counts = np.bincount(idx.reshape(-1), minlength=cfg.E)
        assert counts.min() > 0                                  # every expert's gradient is exercised
