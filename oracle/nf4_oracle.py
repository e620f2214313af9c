"""CPU oracle for 4-bit NormalFloat (NF4) expert base weights -- TEST
INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
import this module.  It shares no code with the CUDA path and imports nothing
from it.

Source: the pages' QLoRA variant of the fine-tuning path.  The Unsloth 2026
wiki page lists 4-bit QLoRA for the Qwen3 MoE family (section "supported
models and 2026 changes", model table) and names LoRA/QLoRA as Unsloth Core's
interface; the GPU MODE lecture 32 notes ("Unsloth -- Faster, Lower-Memory LLM
Fine-Tuning", open questions, the FP8 MMA item) name QLoRA's NF4 base next to
FP8 MMA.  The pages name the format but do not define it.  Read here as QLoRA's published NormalFloat data type (Dettmers et
al., "QLoRA: Efficient Finetuning of Quantized LLMs", 2023, section 3 "4-bit
NormalFloat quantization"):

* the 16 code values are quantiles of the standard normal distribution,
  normalised to [-1, 1]: 8 positive values at probabilities evenly spaced
  from delta down to 1/2 (1/2 itself excluded), 7 negative values mirrored
  from probabilities evenly spaced the same way in 7 steps, and an exact
  zero; delta = 1 - (1/32 + 1/30) / 2, so that the outermost quantile is
  finite.  Code i is the i-th smallest value (code 7 is 0, code 0 is -1,
  code 15 is +1); the values are rounded to float32 once;
* block-wise absmax scaling: each run of 64 consecutive elements of a row
  (the innermost, contiguous dimension) has one float32 scale, its largest
  absolute value; no double quantisation of the scales;
* each element is coded by the code value nearest to w / absmax, both
  computed in float32 (ties to the lower code); an all-zero block has
  absmax 0 and every code 7;
* two codes per byte, the element with the even column index in the low
  nibble;
* the dequantised weight is T[code] * absmax computed in float32 and rounded
  to bf16 (nearest even): the tensor cores take bf16 operands, so this bf16
  value is the base weight the layer computes with.

Parity pins: tests/test_oracle_nf4.py (the code values against the normal CDF
evaluated with math.erf and against the published NF4 values, a block of
known codes with its packed bytes, nearest-code and error-bound invariants,
quantise(dequantise(codes)) == codes, planted slips).
"""
from __future__ import annotations

import numpy as np

BLOCK = 64
NF4_DELTA = 1.0 - 0.5 * (1.0 / 32.0 + 1.0 / 30.0)
ZERO_CODE = 7


def nf4_codebook() -> np.ndarray:
    """The 16 NF4 code values, ascending, float32."""
    from scipy.stats import norm
    positive = norm.ppf(np.linspace(NF4_DELTA, 0.5, 9)[:-1])       # 8 values, largest first
    negative = -norm.ppf(np.linspace(NF4_DELTA, 0.5, 8)[:-1])      # 7 values, smallest first
    v = np.sort(np.concatenate([negative, [0.0], positive]))
    return (v / v.max()).astype(np.float32)


def _f32(a) -> np.ndarray:
    """Weights arrive as torch tensors (bf16) or numpy arrays; bf16 values are exact in float32."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return a.detach().to("cpu", torch.float32).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(a, dtype=np.float32)


def quantize_nf4(W):
    """W: [..., rows, cols] with cols a multiple of 64.  Returns (codes uint8
    [..., rows, cols / 2], two per byte, even column in the low nibble; absmax
    float32 [..., rows, cols / 64])."""
    w = _f32(W)
    *lead, rows, cols = w.shape
    assert cols % BLOCK == 0, "rows must split into blocks of 64"
    blocks = w.reshape(*lead, rows, cols // BLOCK, BLOCK)
    absmax = np.abs(blocks).max(axis=-1).astype(np.float32)
    T = nf4_codebook()
    nonzero = absmax > 0
    with np.errstate(invalid="ignore", divide="ignore"):
        x = (blocks / np.where(nonzero, absmax, np.float32(1))[..., None]).astype(np.float32)
    # nearest code value in float32, the lower code on a tie
    best = np.full(x.shape, np.inf, dtype=np.float32)
    code = np.zeros(x.shape, dtype=np.uint8)
    for c in range(16):
        d = np.abs(x - T[c])
        closer = d < best
        best = np.where(closer, d, best)
        code = np.where(closer, np.uint8(c), code)
    code = np.where(nonzero[..., None], code, np.uint8(ZERO_CODE)).reshape(*lead, rows, cols)
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).astype(np.uint8)
    return packed, absmax


def unpack_nf4(codes) -> np.ndarray:
    """Packed bytes [..., cols / 2] -> one code per element [..., cols]."""
    q = np.asarray(codes, dtype=np.uint8)
    return np.stack([q & 0xF, q >> 4], axis=-1).reshape(*q.shape[:-1], 2 * q.shape[-1])


def dequantize_nf4(codes, absmax) -> np.ndarray:
    """Dequantised base weights (float64 holding bf16 values): T[code] * absmax in
    float32, rounded to bf16."""
    import torch
    c = unpack_nf4(codes)
    s = np.repeat(np.asarray(absmax, dtype=np.float32), BLOCK, axis=-1)
    prod = (nf4_codebook()[c] * s).astype(np.float32)
    return torch.from_numpy(prod).to(torch.bfloat16).to(torch.float64).numpy()
