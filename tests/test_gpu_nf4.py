"""NF4 (4-bit NormalFloat) expert base weights: the device quantiser against the
oracle's (bit for bit), and the NF4 layer against the bf16 layer run on the
dequantised weights (bit for bit: the tensor cores see the same bf16 values), plus
the fp64 oracle on the dequantised weights (tolerance)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as orc
from oracle import nf4_oracle as nf
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
        for wname in ("W_gu", "W_d"):
            W = mi.make_tensor(cfg, wname, 0, "cuda" if name != "tiny" else "cpu").cuda()
            W[0, 1, 64:128] = 0                             # an all-zero block
            W[-1, 5, 7] = 300.0                             # a large outlier
            W[-1, 6, :64] *= 2.0 ** -120                    # a block whose absmax is an fp32 subnormal
            Wq, am = moe.moe_quantize_nf4(W)
            torch.cuda.synchronize()
            for e in (0, W.shape[0] - 1):
                codes, absmax = nf.quantize_nf4(W[e].cpu())
                assert np.array_equal(Wq[e].cpu().numpy(), codes), (name, wname, e)
                # the device stores the scales block-major: [cols / 64, rows]
                assert np.array_equal(am[e].t().cpu().numpy().view(np.uint32), absmax.view(np.uint32)), (name, wname, e)


# Every NF4 launch runs on SM pairs.  The bf16 reference runs on single-CTA tiles for the
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


def _oracle_dequantized(ts, wq):
    """The oracle's codes and scales equal the device's; its dequantised weights (bf16) are
    the reference the NF4 layer must reproduce."""
    deq = {}
    for name_w, qn, sn in (("W_gu", "W4_gu", "m_gu"), ("W_d", "W4_d", "m_d")):
        codes, absmax = nf.quantize_nf4(ts[name_w].cpu())
        assert np.array_equal(wq[qn].cpu().numpy(), codes)
        assert np.array_equal(wq[sn].transpose(-1, -2).cpu().numpy(), absmax)
        deq[name_w] = torch.tensor(nf.dequantize_nf4(codes, absmax)).to(torch.bfloat16).cuda()
    return deq


def _run_both(cfg, idx, w, ts, deq, wq):
    import moe_expert_dispatch_stable_gb300 as moe
    d = moe.Dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r, cfg.scale)
    ti, tw = torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()
    ref = moe.MoELoRALayer(d, {**ts, **deq})
    q4 = moe.MoELoRALayer(d, wq)
    g_ref = ref.step(ti, tw, ts["x"], ts["dy"])
    g_q4 = q4.step(ti, tw, ts["x"], ts["dy"])
    torch.cuda.synchronize()
    assert int(q4.dev_status.item()) == 0 and int(ref.dev_status.item()) == 0
    return ref, q4, g_ref, g_q4


@pytest.mark.parametrize("name", list(CASES))
def test_nf4_layer_is_bit_identical_to_bf16_on_dequantized_weights(name):
    import moe_expert_dispatch_stable_gb300 as moe
    cfg = CASES[name]
    idx, w, ts = make_case(cfg, seed=2)
    wq = moe.quantize_expert_weights(ts, fmt="nf4")
    deq = _oracle_dequantized(ts, wq)
    ref, q4, g_ref, g_q4 = _run_both(cfg, idx, w, ts, deq, wq)
    assert torch.equal(q4.y, ref.y)
    for a, b in zip(g_q4, g_ref):
        assert torch.equal(a, b)
    assert torch.equal(q4.d_topk_w, ref.d_topk_w)
    # and against the fp64 oracle with the dequantised weights
    c = {k: v.cpu() for k, v in {**ts, **deq}.items()}
    wts = [c[n] for n in WEIGHT_NAMES]
    assert_close("y", to64(q4.y), orc.lora_fwd(c["x"], idx, w, *wts, cfg.scale))


@pytest.mark.parametrize("name", ["ragged_bf16_single_cta", "pairs_ragged"])
def test_nf4_extreme_block_scales_bit_identical(name):
    """Blocks whose absmax is far from 1: large (2^20), an fp32 subnormal (the products
    T[code] * absmax are subnormal too), and all-zero blocks -- still bit-identical to the
    bf16 layer on the dequantised weights."""
    import moe_expert_dispatch_stable_gb300 as moe
    cfg = CASES[name]
    idx, w, ts = make_case(cfg, seed=5)
    ts = dict(ts)
    W_gu, W_d = ts["W_gu"].clone(), ts["W_d"].clone()
    W_gu[:, 0:8, 0:64] *= 2.0 ** 20                      # a large gate block in 8 rows
    W_gu[:, 8:16, cfg.I:cfg.I + 64] *= 2.0 ** -125        # tiny up blocks
    W_gu[:, 16, 64:128] = 0
    W_d[:, 3, 64:128] *= 2.0 ** 20
    W_d[:, 5:7, 0:64] *= 2.0 ** -126
    ts["W_gu"], ts["W_d"] = W_gu, W_d
    wq = moe.quantize_expert_weights(ts, fmt="nf4")
    torch.cuda.synchronize()
    assert float(wq["m_gu"][:, cfg.I // 64, 8:16].max()) < 2.0 ** -126
    deq = _oracle_dequantized(ts, wq)
    ref, q4, g_ref, g_q4 = _run_both(cfg, idx, w, ts, deq, wq)
    assert bool(torch.isfinite(ref.y.float()).all())
    assert torch.equal(q4.y, ref.y)
    for a, b in zip(g_q4, g_ref):
        assert torch.equal(a, b)


def _torch_dequantize(Wq, am, T):
    """Per expert on the device: codes -> T[code] (float32) * absmax -> bf16 (the definition,
    one expert at a time to bound the memory of the index tensors)."""
    out = torch.empty(Wq.shape[:-1] + (2 * Wq.shape[-1],), dtype=torch.bfloat16, device=Wq.device)
    for e in range(Wq.shape[0]):
        q = Wq[e].to(torch.int64)
        c = torch.stack([q & 15, q >> 4], dim=-1).reshape(q.shape[0], -1)
        out[e] = (T[c] * am[e].t().repeat_interleave(64, dim=-1)).to(torch.bfloat16)
    return out


def test_nf4_full_size_deepseek_shape_bit_identical():
    """The HBM-bound workload a 4-bit base is for: 256 experts, H = 7168, 128 rows per expert."""
    import moe_expert_dispatch_stable_gb300 as moe
    cfg = mi.CONFIGS["dsv3"]
    idx, w, ts = make_case(cfg, seed=0)
    wq = moe.quantize_expert_weights(ts, fmt="nf4")
    torch.cuda.synchronize()
    d = moe.Dims(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, cfg.r, cfg.scale)
    ti, tw = torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()
    q4 = moe.MoELoRALayer(d, wq)
    g_q4 = [g.clone() for g in q4.step(ti, tw, ts["x"], ts["dy"])]
    y_q4 = q4.y.clone()
    torch.cuda.synchronize()
    assert int(q4.dev_status.item()) == 0
    del q4
    T = torch.tensor(nf.nf4_codebook(), device="cuda")
    bf = dict(ts)
    for name, qn, sn in (("W_gu", "W4_gu", "m_gu"), ("W_d", "W4_d", "m_d")):
        bf[name] = _torch_dequantize(wq[qn], wq[sn], T)
    del wq
    ref = moe.MoELoRALayer(d, bf)
    g_ref = ref.step(ti, tw, ts["x"], ts["dy"])
    torch.cuda.synchronize()
    assert torch.equal(y_q4, ref.y)
    for a, b in zip(g_q4, g_ref):
        assert torch.equal(a, b)
