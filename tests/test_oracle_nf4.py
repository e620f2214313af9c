"""Pins for the NF4 (4-bit NormalFloat) weight quantiser of the oracle (no GPU).

Each pin checks the oracle against something other than itself: the normal CDF
evaluated with math.erf (not the inverse CDF the oracle calls), the NF4 values
published with QLoRA, a block whose codes are known by construction, and
invariants of nearest-value coding.  The last test plants plausible slips in the
oracle and checks that a pin catches each."""
import math

import numpy as np
import pytest
import torch

from oracle import nf4_oracle as nf


def _phi(x: float) -> float:
    return 0.5 * (1.0 + math.erf(x / math.sqrt(2.0)))


def _phi_inv(p: float) -> float:
    lo, hi = 0.0, 10.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if _phi(mid) < p:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def test_codebook_shape_order_and_fixed_points():
    T = nf.nf4_codebook()
    assert T.dtype == np.float32 and T.shape == (16,)
    assert np.all(np.diff(T) > 0)
    assert T[0] == -1.0 and T[15] == 1.0 and T[nf.ZERO_CODE] == 0.0
    assert np.sum(T < 0) == 7 and np.sum(T > 0) == 8


def test_codebook_values_are_normal_quantiles():
    """Phi(T[i] * q) is the i-th probability of the construction, with q the quantile
    at delta; Phi from math.erf and q by bisection on it."""
    T = nf.nf4_codebook().astype(np.float64)
    delta = 1.0 - 0.5 * (1.0 / 32.0 + 1.0 / 30.0)
    q = _phi_inv(delta)
    for i in range(8):                       # positive side: 8 steps from delta towards 1/2
        p = delta - i * (delta - 0.5) / 8
        assert abs(_phi(T[15 - i] * q) - p) < 1e-7, (i, _phi(T[15 - i] * q), p)
    for i in range(7):                       # negative side: 7 steps, mirrored
        p = delta - i * (delta - 0.5) / 7
        assert abs(_phi(-T[i] * q) - p) < 1e-7, (i, _phi(-T[i] * q), p)


# NF4 values as published with QLoRA (Dettmers et al. 2023), to four decimals
PUBLISHED_NF4 = [-1.0, -0.6962, -0.5251, -0.3949, -0.2844, -0.1848, -0.0911, 0.0,
                 0.0796, 0.1609, 0.2461, 0.3379, 0.4407, 0.5626, 0.7230, 1.0]


def test_codebook_matches_published_values():
    np.testing.assert_allclose(nf.nf4_codebook(), PUBLISHED_NF4, rtol=0, atol=1e-4)


def _known_block_weights(perm, shift):
    """A 64-element row block whose values are bf16(T[c]) * 2^shift for codes `perm`
    (a multiple of the 16 codes, so +-1 is in it and absmax is exactly 2^shift)."""
    T = nf.nf4_codebook()
    v = torch.tensor(T[perm]).to(torch.bfloat16).double().numpy() * 2.0 ** shift
    return v


def test_known_codes_and_packing():
    rng = np.random.default_rng(3)
    perms = [np.tile(np.arange(16), 4), np.tile(np.arange(16)[::-1], 4), rng.permutation(np.tile(np.arange(16), 4))]
    shifts = [0, -7, 5]
    W = np.stack([np.concatenate([_known_block_weights(p, s) for p, s in zip(perms, shifts)])])[None]  # [1,1,192]
    codes, absmax = nf.quantize_nf4(torch.tensor(W).to(torch.bfloat16))
    assert codes.shape == (1, 1, 96) and absmax.shape == (1, 1, 3)
    np.testing.assert_array_equal(absmax[0, 0], [2.0 ** s for s in shifts])
    want = np.concatenate(perms).astype(np.uint8)
    np.testing.assert_array_equal(nf.unpack_nf4(codes)[0, 0], want)
    # two codes per byte, the even column in the low nibble
    np.testing.assert_array_equal(codes[0, 0], want[0::2] + 16 * want[1::2])
    assert codes[0, 0, 0] == 0x10 and codes[0, 0, 1] == 0x32        # codes 0,1 and 2,3


def test_zero_block_and_block_extremes():
    rng = np.random.default_rng(4)
    W = rng.standard_normal((2, 4, 128)) * 0.05
    W[1, 2, 64:] = 0.0                                          # an all-zero block
    Wb = torch.tensor(W).to(torch.bfloat16)
    codes, absmax = nf.quantize_nf4(Wb)
    c = nf.unpack_nf4(codes)
    assert absmax[1, 2, 1] == 0 and np.all(c[1, 2, 64:] == nf.ZERO_CODE)
    w = Wb.float().numpy().reshape(2, 4, 2, 64)
    cb = c.reshape(2, 4, 2, 64)
    for m, r, b in np.ndindex(2, 4, 2):
        if absmax[m, r, b] == 0:
            continue
        i = np.argmax(np.abs(w[m, r, b]))
        assert absmax[m, r, b] == abs(w[m, r, b, i])
        assert cb[m, r, b, i] == (15 if w[m, r, b, i] > 0 else 0)   # w / absmax = +-1 exactly


def test_codes_are_nearest_and_error_is_bounded():
    rng = np.random.default_rng(5)
    W = rng.standard_normal((3, 6, 256)) * np.exp(rng.uniform(-6, 2, (3, 6, 1)))
    Wb = torch.tensor(W).to(torch.bfloat16)
    codes, absmax = nf.quantize_nf4(Wb)
    T = nf.nf4_codebook().astype(np.float64)
    w = Wb.double().numpy()
    s = np.repeat(absmax.astype(np.float64), 64, axis=-1)
    x = w / s                                                    # exact ratio in float64
    c = nf.unpack_nf4(codes)
    d_code = np.abs(x - T[c])
    d_best = np.abs(x[..., None] - T).min(axis=-1)
    # the chosen value is the nearest one, up to the float32 rounding of w / absmax
    assert np.all(d_code <= d_best + 2e-7)
    # and within half the largest gap between neighbouring code values
    assert np.all(d_code <= 0.5 * np.diff(T).max() + 1e-7)
    deq = nf.dequantize_nf4(codes, absmax)
    assert np.array_equal(torch.tensor(deq).to(torch.bfloat16).double().numpy(), deq)   # bf16 values
    assert np.all(np.abs(deq - w) <= s * (0.5 * np.diff(T).max() + 2.0 ** -8) + 1e-30)


def test_quantize_of_dequantized_weights_returns_the_codes():
    """absmax is a bf16 value, so dequantising a block keeps its absmax, and each
    dequantised value stays nearest to its own code value."""
    rng = np.random.default_rng(6)
    W = torch.tensor(rng.standard_normal((2, 5, 192)) * 0.03).to(torch.bfloat16)
    codes, absmax = nf.quantize_nf4(W)
    deq = torch.tensor(nf.dequantize_nf4(codes, absmax)).to(torch.bfloat16)
    codes2, absmax2 = nf.quantize_nf4(deq)
    np.testing.assert_array_equal(codes2, codes)
    np.testing.assert_array_equal(absmax2, absmax)


def test_planted_slips_are_caught(monkeypatch):
    """A swapped nibble order, a table missing its renormalisation, and round-down
    instead of nearest: each fails one of the pins above."""
    real_q = nf.quantize_nf4

    def swapped_nibbles(W):
        q, a = real_q(W)
        return ((q >> 4) | (q << 4)).astype(np.uint8), a

    monkeypatch.setattr(nf, "quantize_nf4", swapped_nibbles)
    with pytest.raises(AssertionError):
        test_known_codes_and_packing()
    monkeypatch.undo()

    real_T = nf.nf4_codebook

    def unnormalised():
        from scipy.stats import norm
        pos = norm.ppf(np.linspace(nf.NF4_DELTA, 0.5, 9)[:-1])
        neg = -norm.ppf(np.linspace(nf.NF4_DELTA, 0.5, 8)[:-1])
        return np.sort(np.concatenate([neg, [0.0], pos])).astype(np.float32)

    monkeypatch.setattr(nf, "nf4_codebook", unnormalised)
    with pytest.raises(AssertionError):
        test_codebook_shape_order_and_fixed_points()
    monkeypatch.undo()
    assert nf.nf4_codebook is real_T

    def round_down(W):
        w = nf._f32(W)
        *lead, rows, cols = w.shape
        blocks = w.reshape(*lead, rows, cols // 64, 64)
        a = np.abs(blocks).max(axis=-1).astype(np.float32)
        x = blocks / np.where(a > 0, a, 1)[..., None]
        T = nf.nf4_codebook()
        c = np.clip(np.searchsorted(T, x, side="right") - 1, 0, 15).astype(np.uint8).reshape(*lead, rows, cols)
        return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8), a

    monkeypatch.setattr(nf, "quantize_nf4", round_down)
    with pytest.raises(AssertionError):
        test_codes_are_nearest_and_error_is_bounded()
