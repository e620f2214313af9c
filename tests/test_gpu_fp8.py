"""FP8 (e4m3) expert base weights: the device quantiser against the oracle's (bit
for bit), and the FP8 layer against the bf16 layer run on the dequantised
weights (bit for bit: the tensor cores see the same bf16 values), plus the fp64
oracle on the dequantised weights (tolerance)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as orc
from tests.gpu_common import WEIGHT_NAMES, assert_close, make_case, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def test_quantizer_bit_exact_against_oracle():
    import moe_expert_dispatch_stable_gb300 as moe
    for name in ("tiny", "gptoss20b"):
        cfg = mi.CONFIGS[name]
        W = mi.make_tensor(cfg, "W_d", 0, "cuda" if name != "tiny" else "cpu").cuda()
        W[0, :, 3] = 0                                  # an all-zero column
        W[-1, 5, 7] = 300.0                             # a large outlier
        Wq, sc = moe.moe_quantize_fp8(W)
        torch.cuda.synchronize()
        for e in (0, W.shape[0] - 1):
            codes, scales = orc.quantize_fp8(W[e].cpu())
            assert np.array_equal(Wq[e].cpu().numpy(), codes)
            assert np.array_equal(sc[e].cpu().numpy(), scales)


# Every FP8 launch runs on SM pairs.  The bf16 reference runs on single-CTA tiles for the
# first case (about 233 rows per expert) and on SM pairs for the others.
CASES = {
    "ragged_bf16_single_cta": mi.MoEConfig("ragged", T=700, H=256, E=6, k=2, I=320, r=16, alpha=32),
    "pairs_ragged": mi.MoEConfig("pairs", T=1000, H=256, E=4, k=2, I=320, r=16, alpha=32),
    "tiny_r8": mi.CONFIGS["tiny"],
    # ~3 tiles per SM pair: the converters carry their stage parity across tiles and
    # LoRA steps
    "multi_tile": mi.MoEConfig("multitile", T=8192, H=512, E=8, k=2, I=512, r=16, alpha=32),
    # LoRA rank 64: the unconverted LoRA stage carries four 16-deep MMA slices
    "pairs_r64": mi.MoEConfig("pairs_r64", T=1000, H=256, E=4, k=2, I=320, r=64, alpha=128),
    # every token routed to every expert (k = E), rank 32
    "k_equals_e_r32": mi.MoEConfig("keqe", T=400, H=192, E=4, k=4, I=256, r=32, alpha=64),
    # three converter groups for the k = 2560 GEMMs (gate_up forward, down backward), two
    # for the others
    "long_k_three_groups": mi.MoEConfig("longk", T=600, H=2560, E=4, k=2, I=256, r=16, alpha=32),
    # half tiles (64 rows per expert) with k = 2048: three groups except the down forward
    "half_tiles_three_groups": mi.MoEConfig("halfk", T=256, H=2048, E=8, k=2, I=1024, r=16, alpha=32),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fp8_layer_is_bit_identical_to_bf16_on_dequantized_weights(name):
    import moe_expert_dispatch_stable_gb300 as moe
    cfg = CASES[name]
    idx, w, ts = make_case(cfg, seed=2)
    wq = moe.quantize_expert_weights(ts)
    # the oracle's quantiser on the same bf16 weights gives the same codes and scales, and
    # its dequantised weights are the bf16 reference the FP8 layer must reproduce
    deq = {}
    for name_w, qn, sn in (("W_gu", "Wq_gu", "s_gu"), ("W_d", "Wq_d", "s_d")):
        codes, scales = orc.quantize_fp8(ts[name_w].cpu())
        assert np.array_equal(wq[qn].cpu().numpy(), codes) and np.array_equal(wq[sn].cpu().numpy(), scales)
        deq[name_w] = torch.tensor(orc.dequantize_fp8(codes, scales)).to(torch.bfloat16).cuda()
    bf_w = {**ts, **deq}
    d = moe.Dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r, cfg.scale)
    ti, tw = torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()
    ref = moe.MoELoRALayer(d, bf_w)
    q8 = moe.MoELoRALayer(d, wq)
    g_ref = ref.step(ti, tw, ts["x"], ts["dy"])
    g_q8 = q8.step(ti, tw, ts["x"], ts["dy"])
    torch.cuda.synchronize()
    assert int(q8.dev_status.item()) == 0
    assert torch.equal(q8.y, ref.y)
    for a, b in zip(g_q8, g_ref):
        assert torch.equal(a, b)
    assert torch.equal(q8.d_topk_w, ref.d_topk_w)
    # and against the fp64 oracle with the dequantised weights
    c = {k: v.cpu() for k, v in {**ts, **deq}.items()}
    wts = [c[n] for n in WEIGHT_NAMES]
    assert_close("y", to64(q8.y), orc.lora_fwd(c["x"], idx, w, *wts, cfg.scale))



@pytest.mark.parametrize("name", ["ragged_bf16_single_cta", "pairs_ragged"])
def test_fp8_extreme_column_scales_bit_identical(name):
    """Columns whose power-of-two scale is far from 1: above 2^7 (the dequantising
    multiply is split in two), below fp32's normal range (a subnormal scale), and tiny
    enough that code * scale rounds in bf16 -- the FP8 layer still matches the bf16 layer
    on the dequantised weights bit for bit."""
    import moe_expert_dispatch_stable_gb300 as moe
    cfg = CASES[name]
    idx, w, ts = make_case(cfg, seed=5)
    ts = dict(ts)
    W_gu, W_d = ts["W_gu"].clone(), ts["W_d"].clone()
    W_gu[:, :, 0:8] *= 2.0 ** 26                         # gate columns: scale > 2^7
    W_gu[:, :, cfg.I + 8:cfg.I + 16] *= 2.0 ** -120      # up columns: scale below 2^-126
    W_d[:, :, 3] *= 2.0 ** 26
    W_d[:, :, 5:7] *= 2.0 ** -125
    ts["W_gu"], ts["W_d"] = W_gu, W_d
    wq = moe.quantize_expert_weights(ts)
    torch.cuda.synchronize()
    assert float(wq["s_gu"][:, 0:8].min()) > 2.0 ** 7
    assert float(wq["s_gu"][:, cfg.I + 8:cfg.I + 16].max()) < 2.0 ** -126
    bf = dict(ts)
    for name_w, qn, sn in (("W_gu", "Wq_gu", "s_gu"), ("W_d", "Wq_d", "s_d")):
        codes, scales = orc.quantize_fp8(ts[name_w].cpu())
        assert np.array_equal(wq[qn].cpu().numpy(), codes) and np.array_equal(wq[sn].cpu().numpy(), scales)
        bf[name_w] = (wq[qn].view(torch.float8_e4m3fn).float() * wq[sn][:, None, :]).to(torch.bfloat16)
    d = moe.Dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r, cfg.scale)
    ti, tw = torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()
    ref = moe.MoELoRALayer(d, bf)
    q8 = moe.MoELoRALayer(d, wq)
    g_ref = ref.step(ti, tw, ts["x"], ts["dy"])
    g_q8 = q8.step(ti, tw, ts["x"], ts["dy"])
    torch.cuda.synchronize()
    assert int(q8.dev_status.item()) == 0
    assert bool(torch.isfinite(ref.y.float()).all())
    assert torch.equal(q8.y, ref.y)
    for a, b in zip(g_q8, g_ref):
        assert torch.equal(a, b)

def test_fp8_full_size_deepseek_shape_bit_identical():
    """The HBM-bound workload FP8 weights are for: 256 experts, H = 7168, 128 rows per expert."""
    import moe_expert_dispatch_stable_gb300 as moe
    cfg = mi.CONFIGS["dsv3"]
    idx, w, ts = make_case(cfg, seed=0)
    wq = moe.quantize_expert_weights(ts)
    torch.cuda.synchronize()
    d = moe.Dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r, cfg.scale)
    ti, tw = torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()
    q8 = moe.MoELoRALayer(d, wq)
    g_q8 = [g.clone() for g in q8.step(ti, tw, ts["x"], ts["dy"])]
    y_q8 = q8.y.clone()
    del q8
    # dequantise on the device with torch (codes -> e4m3 -> float * scale -> bf16, exact)
    bf = dict(ts)
    for name, qn, sn in (("W_gu", "Wq_gu", "s_gu"), ("W_d", "Wq_d", "s_d")):
        bf[name] = (wq[qn].view(torch.float8_e4m3fn).float() * wq[sn][:, None, :]).to(torch.bfloat16)
    del wq
    ref = moe.MoELoRALayer(d, bf)
    g_ref = ref.step(ti, tw, ts["x"], ts["dy"])
    torch.cuda.synchronize()
    assert torch.equal(y_q8, ref.y)
    for a, b in zip(g_q8, g_ref):
        assert torch.equal(a, b)
