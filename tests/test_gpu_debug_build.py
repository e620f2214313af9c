"""The debug build of the library (MOE_DEBUG=1, libmoe_lora_gb300_debug.so).

Its kernels check every index they read from a routing buffer -- perm in the gathers,
inv_perm in the combines, offsets / tile_offsets in the grouped GEMMs and LoRA
reductions -- before using it.  On valid input it computes exactly what the release
build computes; an index out of range sets MOE_DEV_BAD_INDEX in the status word and the
access is skipped (no trap, no fault: the context stays usable).  The corrupted-routing
cases run on the debug build only: the release build trusts moe_route's outputs.
"""
import pytest
import torch

import moe_inputs as mi
from tests.gpu_common import make_case

pytestmark = pytest.mark.gpu

CASES = {
    "ragged": mi.MoEConfig("ragged", T=700, H=256, E=6, k=2, I=320, r=16, alpha=32),
    # >= 384 rows per expert: the expert GEMMs run on SM pairs
    "pairs_skew": mi.MoEConfig("pairs_skew", T=2000, H=128, E=8, k=2, I=192, r=8, alpha=16, zipf_s=1.2),
}


@pytest.fixture(scope="module")
def debug_path():
    import __graft_entry__
    from moe_expert_dispatch_stable_gb300 import build
    __graft_entry__.build()
    torch.cuda.set_device(0)
    return build.build(debug=True)


def _layer(cfg, seed=0):
    import moe_expert_dispatch_stable_gb300 as moe
    idx, w, ts = make_case(cfg, seed=seed)
    layer = moe.MoELoRALayer(moe.Dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r, cfg.scale), ts)
    return layer, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), ts


def _outputs(layer):
    return [layer.y.clone(), layer.dx.clone(), layer.d_topk_w.clone()] + [g.clone() for g in layer.grads]


@pytest.mark.parametrize("name", list(CASES))
def test_debug_build_is_bit_identical_on_valid_input(debug_path, name):
    from moe_expert_dispatch_stable_gb300 import binding
    layer, ti, tw, ts = _layer(CASES[name])
    layer.step(ti, tw, ts["x"], ts["dy"])
    torch.cuda.synchronize()
    ref = _outputs(layer)
    with binding.using_library(debug_path):
        layer.step(ti, tw, ts["x"], ts["dy"])
        torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    for a, b in zip(ref, _outputs(layer)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("field,index,value", [
    ("perm", 5, 10 ** 7), ("perm", -1, -3),             # the gathers (x, weighted dy, d topk_w)
    ("inv_perm", 3, 10 ** 7), ("inv_perm", 0, -1),      # the combines
    ("offsets", 2, 10 ** 7), ("offsets", -1, 0),         # the grouped GEMMs and LoRA reductions
    ("tile_offsets", 1, 10 ** 6),                        # the single-CTA tile scheduler
])
def test_debug_build_flags_and_skips_bad_routing_indices(debug_path, name, field, index, value):
    import moe_expert_dispatch_stable_gb300 as moe
    from moe_expert_dispatch_stable_gb300 import binding
    layer, ti, tw, ts = _layer(CASES[name], seed=1)
    with binding.using_library(debug_path):
        layer.route(ti, tw)
        getattr(layer.rt, field)[index] = value
        layer.dev_status.zero_()
        layer.forward(ts["x"])
        layer.backward(ts["dy"])
        torch.cuda.synchronize()                            # returns: nothing faulted
        status = int(layer.dev_status.item())
    # (tile_offsets: the SM-pair expert GEMMs derive their tiles from the offsets, but the
    # rank-r projections run single-CTA tiles and read them in every layer)
    assert status & moe.binding.MOE_DEV_BAD_INDEX, (field, index, status)
    # the context is still usable: a clean step of the release build on the same buffers
    layer.dev_status.zero_()
    layer.step(ti, tw, ts["x"], ts["dy"])
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
