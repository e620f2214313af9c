"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every mbarrier wait inside the tensor-core kernels is bounded.  A wait that runs
out sets MOE_DEV_TIMEOUT; the kernel stops issuing work, waits until the copies
and MMAs it already issued have landed, frees its TMEM and returns, so the
context stays usable.  moe_diag_force_timeout makes a chosen launch do exactly
that: its epilogue waits on an mbarrier that nothing arrives on, with a 1 ms
limit, and its other roles then run out of work to wait for.  Each of the ten
single-CTA tensor-core launches of a step (four forward, six backward) is made
to fail in turn; the call returns, the flag is set, and the next step on the
same buffers gives bit for bit the results of a step before the failure.
"""
import pytest
import torch

import moe_inputs as mi

pytestmark = pytest.mark.gpu

LAUNCHES_PER_STEP = 10     # proj XA, gate_up, proj HA, down | proj G, down bwd, wgrad, proj Gg, gate_up bwd, wgrad
CASES = {
    "tiny": mi.CONFIGS["tiny"],
    # about 3.4 gate_up tiles per CTA on 152 SMs: the MMA issuer stops at its third tile while
    # the producer has filled the ring, so unconsumed loads are in flight when the waits give up
    "deep": mi.MoEConfig("deep", T=16384, H=128, E=64, k=1, I=512, r=16, alpha=32),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("name", list(CASES))
def test_forced_wait_timeout_sets_flag_and_leaves_context_usable(name):
    import moe_expert_dispatch_stable_gb300 as moe
    cfg = CASES[name]
    assert cfg.T * cfg.k < 384 * cfg.E                 # single-CTA tiles: the launches the hook counts
    idx, w = mi.make_routing(cfg, 0)
    ts = {n: mi.make_tensor(cfg, n, 0, "cpu").cuda() for n in mi.TENSOR_NAMES}
    d = moe.Dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r, cfg.scale)
    layer = moe.MoELoRALayer(d, ts)
    ti, tw = torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()

    def outputs():
        return [layer.y.clone(), layer.dx.clone()] + [g.clone() for g in layer.grads]

    layer.step(ti, tw, ts["x"], ts["dy"])
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    ref = outputs()
    try:
        for i in range(LAUNCHES_PER_STEP):
            layer.dev_status.zero_()
            moe.moe_diag_force_timeout(i, 1_000_000)
            layer.step(ti, tw, ts["x"], ts["dy"])
            torch.cuda.synchronize()                    # returns: no fault, no hang
            status = int(layer.dev_status.item())
            assert status & moe.binding.MOE_DEV_TIMEOUT, (name, i, status)
            assert not status & moe.binding.MOE_DEV_BAD_EXPERT_ID
            layer.dev_status.zero_()
            layer.step(ti, tw, ts["x"], ts["dy"])
            torch.cuda.synchronize()
            assert int(layer.dev_status.item()) == 0, (name, i)
            for a, b in zip(ref, outputs()):
                assert torch.equal(a, b), (name, i)
    finally:
        moe.moe_diag_force_timeout(-1, 0)


def test_hook_outside_a_step_counts_only_single_cta_launches():
    """Armed past the last launch of a step, the hook fires in the next step."""
    import moe_expert_dispatch_stable_gb300 as moe
    cfg = CASES["tiny"]
    idx, w = mi.make_routing(cfg, 1)
    ts = {n: mi.make_tensor(cfg, n, 1, "cpu").cuda() for n in mi.TENSOR_NAMES}
    layer = moe.MoELoRALayer(moe.Dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r, cfg.scale), ts)
    ti, tw = torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()
    try:
        moe.moe_diag_force_timeout(LAUNCHES_PER_STEP + 1, 1_000_000)   # the second launch of the next step
        layer.step(ti, tw, ts["x"], ts["dy"])
        torch.cuda.synchronize()
        assert int(layer.dev_status.item()) == 0
        layer.step(ti, tw, ts["x"], ts["dy"])
        torch.cuda.synchronize()
        assert int(layer.dev_status.item()) & moe.binding.MOE_DEV_TIMEOUT
    finally:
        moe.moe_diag_force_timeout(-1, 0)
