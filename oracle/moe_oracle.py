"""CPU oracle for the LoRA-fine-tuned MoE expert layer -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  It shares no code with the CUDA path
and imports nothing from it.

Everything here is plain numpy in float64, written to be checked by eye
against the pages:

* routing -- "Unsloth and NVIDIA" blog post (d9249.github.io, "How to make
  LLM training faster with Unsloth and NVIDIA" write-up), section
  "core idea / structure / how it works", GPT-OSS MoE routing paragraphs: the
  old path asks ``torch.where(router_indices == e)`` once per expert; the new
  path flattens the top-k assignment, stable-sorts it by expert id, bincounts
  it once and slices by offsets.  The routing logic itself does not change,
  so both give the same grouping.  The oracle uses the per-expert ``where``
  form (one query per expert) and builds perm / counts / offsets from it.
* forward / backward -- Unsloth 2026 wiki page ("GRPO, MoE and memory
  efficient fine-tuning"), section "Optimisation 3: grouped_mm and
  Split-LoRA for MoE training": all experts' weights stacked in one tensor,
  group sizes equal to the routing counts, and the LoRA delta either merged
  into W ("standard PEFT: x -> (W + BA)") or applied separately (Split-LoRA),
  the two being mathematically identical.  The oracle uses the merged form
  M = W + s * A B in fp64; the CUDA path uses the split form.
* SwiGLU -- named (not defined) among the hand-written kernels in the GPU MODE
  lecture 32 notes ("Unsloth -- Faster, Lower-Memory LLM Fine-Tuning").  Read
  here as h = silu(g) * u with g the first I columns of the gate_up product
  and u the last I columns; silu(z) = z * sigmoid(z).
* routing-weighted combine -- same wiki section, "bottleneck of the existing
  implementation": every expert's output is weighted by the token's routing
  weight for that expert and the outputs are summed.  Read as y[t] =
  sum_j w[t,j] * f_{e(t,j)}(x[t]) (the weight multiplies the expert output).
* backward -- the GPU MODE lecture's principle "start from the exact math":
  the gradient of each step is derived by hand (here: chain rule through the
  merged matrices, below), not by autograd.
* router -- the step in front of the routing in every workload: softmax over
  the E router logits of a token, then the k largest probabilities (no
  renormalisation, ties to the lower expert index); its backward is the
  softmax VJP with the selection held fixed, fed by dL/dw[t,j] = <dy[t],
  unweighted expert output> (y is linear in the routing weights).

Layouts follow the C ABI: x [T,H]; W_gu [E,H,2I]; W_d [E,I,H]; A_gu [E,r,H]
(= A^T, PEFT lora_A layout); B_gu [E,r,2I]; A_d [E,r,I]; B_d [E,r,H].
In math form A_math = A_stored^T (in x r) and B_math = B_stored (r x out).

Parity pins: see tests/test_oracle.py (invariants, library sort, brute force,
split == merged, B = 0, E = 1 dense MLP, finite differences, a hand-worked
golden case) and tests/test_oracle_router.py (library top-k, torch autograd
of the softmax, exact directional derivative in w, finite differences of the
composed router + layer).  No numeric example is printed on the pages.
"""
from __future__ import annotations

import numpy as np


def _f64(a):
    """Inputs arrive as torch tensors (often bf16) or numpy arrays; the oracle
    works on their exact values in float64."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return a.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(a, dtype=np.float64)


def _i64(a):
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return a.detach().to("cpu", torch.int64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(a, dtype=np.int64)


# --------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------
def route(topk_idx, E: int):
    """Group the T*k routed slots by expert.

    Returns (counts [E], offsets [E+1], perm [T*k], inv_perm [T*k]) as int64.
    perm[p] is the flat slot index t*k + j; the slots of expert e occupy
    perm[offsets[e]:offsets[e+1]] in ascending flat index (the stable order).
    Built from one ``where`` query per expert, the pages' "before" form.
    """
    flat = _i64(topk_idx).reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    counts = np.zeros(E, dtype=np.int64)
    parts = []
    for e in range(E):
        (slots,) = np.where(flat == e)      # ascending flat indices
        counts[e] = slots.size
        parts.append(slots)
    perm = np.concatenate(parts) if parts else np.zeros(0, np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    inv_perm = np.empty_like(perm)
    inv_perm[perm] = np.arange(perm.size, dtype=np.int64)
    return counts, offsets, perm.astype(np.int64), inv_perm


def tile_offsets(counts, bm: int):
    """Prefix sum of per-expert tile counts ceil(counts[e] / bm) (scheduler input)."""
    c = _i64(counts)
    t = np.zeros(c.size + 1, dtype=np.int64)
    t[1:] = np.cumsum((c + bm - 1) // bm)
    return t


# --------------------------------------------------------------------------
# expert MLP pieces
# --------------------------------------------------------------------------
def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    return z * sigmoid(z)


def swiglu(gu, I: int):
    """h = silu(g) * u with g = gu[:, :I], u = gu[:, I:]."""
    g, u = gu[:, :I], gu[:, I:]
    return silu(g) * u


def swiglu_bwd(dh, gu, I: int):
    """Hand-derived VJP of swiglu: d/dg [g sig(g) u] = u sig (1 + g (1 - sig));
    d/du = silu(g).  Returns dGU = [dg | du]."""
    g, u = gu[:, :I], gu[:, I:]
    sg = sigmoid(g)
    dg = dh * u * sg * (1.0 + g * (1.0 - sg))
    du = dh * g * sg
    return np.concatenate([dg, du], axis=1)


def merged(W_e, A_e, B_e, scale):
    """Standard-PEFT merged weight W + s * A_math B_math (A stored transposed)."""
    return W_e + scale * (A_e.T @ B_e)


# --------------------------------------------------------------------------
# forward / backward
# --------------------------------------------------------------------------
def _expert_rows(topk_idx, e, token_subset=None):
    t_idx, j_idx = np.where(topk_idx == e)
    if token_subset is not None:
        keep = np.isin(t_idx, token_subset)
        t_idx, j_idx = t_idx[keep], j_idx[keep]
    return t_idx, j_idx


def lora_fwd(x, topk_idx, topk_w, W_gu, A_gu, B_gu, W_d, A_d, B_d, scale,
             token_subset=None):
    """y[t] = sum_j w[t,j] * (swiglu(x[t] M_gu[e]) M_d[e]),  e = topk_idx[t,j],
    with M = W + s * A B merged per expert, fp64.

    token_subset: optional array of token ids; rows of y outside it stay zero."""
    x = _f64(x); w = _f64(topk_w); idx = _i64(topk_idx)
    T, H = x.shape
    E = W_gu.shape[0]
    I = W_d.shape[1]
    y = np.zeros((T, H))
    for e in range(E):
        t_idx, j_idx = _expert_rows(idx, e, token_subset)
        if t_idx.size == 0:
            continue
        M_gu = merged(_f64(W_gu[e]), _f64(A_gu[e]), _f64(B_gu[e]), scale)
        M_d = merged(_f64(W_d[e]), _f64(A_d[e]), _f64(B_d[e]), scale)
        X = x[t_idx]
        h = swiglu(X @ M_gu, I)
        O = h @ M_d
        np.add.at(y, t_idx, w[t_idx, j_idx][:, None] * O)
    return y


def lora_bwd(dy, x, topk_idx, topk_w, W_gu, A_gu, B_gu, W_d, A_d, B_d, scale,
             token_subset=None, expert_subset=None):
    """Gradients of L = <dy, y> w.r.t. x and the four LoRA factors (base W frozen).

    Per expert e with merged M_gu, M_d (fp64):
      X = x[t(e)], GU = X M_gu, h = swiglu(GU), dO = w * dy[t(e)]
      dh = dO M_d^T;  dGU = swiglu_bwd(dh, GU);  dx[t] += dGU M_gu^T
      dM_gu = X^T dGU;  dM_d = h^T dO
      M = W + s A_math B  =>  dA_math = s dM B^T, dB = s A_math^T dM
    Stored layouts: dA_stored = (dA_math)^T = s B dM^T, dB_stored = s A_stored dM.

    token_subset restricts dx (rows outside stay 0); expert_subset restricts the
    LoRA gradients (other experts stay 0).  An expert's LoRA gradient always
    uses all of its rows."""
    x = _f64(x); w = _f64(topk_w); idx = _i64(topk_idx); dy = _f64(dy)
    T, H = x.shape
    E = W_gu.shape[0]
    I = W_d.shape[1]
    r = A_gu.shape[1]
    dx = np.zeros((T, H))
    dA_gu = np.zeros((E, r, H)); dB_gu = np.zeros((E, r, 2 * I))
    dA_d = np.zeros((E, r, I)); dB_d = np.zeros((E, r, H))
    for e in range(E):
        want_lora = expert_subset is None or e in set(np.asarray(expert_subset).tolist())
        t_idx, j_idx = _expert_rows(idx, e, None if want_lora else token_subset)
        if t_idx.size == 0:
            continue
        Agu, Bgu = _f64(A_gu[e]), _f64(B_gu[e])
        Ad, Bd = _f64(A_d[e]), _f64(B_d[e])
        M_gu = merged(_f64(W_gu[e]), Agu, Bgu, scale)
        M_d = merged(_f64(W_d[e]), Ad, Bd, scale)
        X = x[t_idx]
        GU = X @ M_gu
        h = swiglu(GU, I)
        dO = w[t_idx, j_idx][:, None] * dy[t_idx]
        dh = dO @ M_d.T
        dGU = swiglu_bwd(dh, GU, I)
        dX = dGU @ M_gu.T
        if token_subset is None:
            np.add.at(dx, t_idx, dX)
        else:
            keep = np.isin(t_idx, token_subset)
            np.add.at(dx, t_idx[keep], dX[keep])
        if want_lora:
            dM_gu = X.T @ dGU          # [H, 2I]
            dM_d = h.T @ dO            # [I, H]
            dA_gu[e] = scale * (Bgu @ dM_gu.T)
            dB_gu[e] = scale * (Agu @ dM_gu)
            dA_d[e] = scale * (Bd @ dM_d.T)
            dB_d[e] = scale * (Ad @ dM_d)
    return dx, dA_gu, dB_gu, dA_d, dB_d


# --------------------------------------------------------------------------
# router (the step in front of the routing, and its gradient)
# --------------------------------------------------------------------------
def router_topk(logits, k: int):
    """Softmax over all E logits, then the k largest probabilities, descending,
    ties to the lower expert index, no renormalisation (the router recipe of
    the workloads).  Softmax is strictly increasing in each logit, so the
    selection is made on the logits themselves and is exact.

    Returns topk_idx [T,k] int64, topk_w [T,k] and the probabilities p [T,E]."""
    z = _f64(logits)
    order = np.argsort(-z, axis=1, kind="stable")[:, :k]
    zc = z - z.max(axis=1, keepdims=True)
    p = np.exp(zc)
    p /= p.sum(axis=1, keepdims=True)
    return order.astype(np.int64), np.take_along_axis(p, order, axis=1), p


def router_bwd(logits, topk_idx, d_topk_w):
    """VJP of topk_w[t,j] = softmax(z[t])[topk_idx[t,j]] with the selection held
    fixed: d p_i / d z_e = p_i (delta_ie - p_e), hence
      dz[t,e] = p_e * (g_e - sum_j d_topk_w[t,j] * topk_w[t,j]),
    with g_e = d_topk_w[t,j] if e = topk_idx[t,j] (else 0)."""
    z = _f64(logits)
    idx = _i64(topk_idx)
    dw = _f64(d_topk_w)
    zc = z - z.max(axis=1, keepdims=True)
    p = np.exp(zc)
    p /= p.sum(axis=1, keepdims=True)
    w = np.take_along_axis(p, idx, axis=1)
    g = np.zeros_like(p)
    np.put_along_axis(g, idx, dw, axis=1)
    return p * (g - (dw * w).sum(axis=1, keepdims=True))


def lora_dtopk_w(dy, x, topk_idx, W_gu, A_gu, B_gu, W_d, A_d, B_d, scale, token_subset=None):
    """Gradient of L = <dy, y> w.r.t. the routing weights: y is linear in them,
    so dL/dw[t,j] = <dy[t], f_e(x[t])> with f_e the unweighted expert output
    (merged weights, fp64).  Slots of tokens outside token_subset stay 0."""
    x = _f64(x); idx = _i64(topk_idx); dy = _f64(dy)
    T = x.shape[0]
    E = W_gu.shape[0]
    I = W_d.shape[1]
    dw = np.zeros(idx.shape)
    for e in range(E):
        t_idx, j_idx = _expert_rows(idx, e, token_subset)
        if t_idx.size == 0:
            continue
        M_gu = merged(_f64(W_gu[e]), _f64(A_gu[e]), _f64(B_gu[e]), scale)
        M_d = merged(_f64(W_d[e]), _f64(A_d[e]), _f64(B_d[e]), scale)
        O = swiglu(x[t_idx] @ M_gu, I) @ M_d
        dw[t_idx, j_idx] = (dy[t_idx] * O).sum(axis=1)
    return dw


# --------------------------------------------------------------------------
# FP8 (e4m3) expert base weights
# --------------------------------------------------------------------------
E4M3_MAX = 448.0


def quantize_fp8(W):
    """Per matrix and column: scale = 2^ceil(log2(amax / 448)) (1 for an all-zero
    column), codes = e4m3 round-to-nearest-even of W / scale.  W: [..., rows, cols].
    Returns (codes uint8 in the e4m3 bit layout, scales float32 [..., cols]).

    With power-of-two scales, W / scale is exact, and code * scale rounded to bf16
    (exact unless the scale is so small that the product falls below bf16's normal
    range) gives a set of bf16 base weights."""
    import torch
    w = _f64(W)
    amax = np.abs(w).max(axis=-2)
    with np.errstate(divide="ignore"):
        e = np.ceil(np.log2(amax / E4M3_MAX))
    scale = np.where(amax > 0, np.exp2(e), 1.0)
    q = torch.tensor(w / scale[..., None, :], dtype=torch.float64).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).numpy(), scale.astype(np.float32)


def dequantize_fp8(codes, scales):
    """Dequantised weights (float64): e4m3 value of each code times its column scale."""
    import torch
    c = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return c * np.asarray(scales, np.float64)[..., None, :]
