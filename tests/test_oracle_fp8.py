"""Pins for the FP8 (e4m3) weight quantiser of the oracle (no GPU)."""
import itertools

import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc


def _e4m3_table():
    """Every finite e4m3 value from its bit layout (1 sign, 4 exponent bits with bias
    7, 3 mantissa bits; exponent field 0 is subnormal; 0x7F / 0xFF are NaN)."""
    vals = {}
    for b in range(256):
        s = -1.0 if b & 0x80 else 1.0
        e = (b >> 3) & 0xF
        m = b & 7
        if (b & 0x7F) == 0x7F:
            continue
        v = s * (m / 8.0) * 2.0 ** -6 if e == 0 else s * (1 + m / 8.0) * 2.0 ** (e - 7)
        vals[b] = v
    return vals


def test_e4m3_table_matches_torch_decoding():
    t = _e4m3_table()
    codes = torch.tensor(list(t.keys()), dtype=torch.uint8)
    dec = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(dec, np.array(list(t.values())))
    assert max(t.values()) == 448.0


def test_codes_are_nearest_e4m3_value_ties_to_even():
    rng = np.random.default_rng(0)
    W = rng.standard_normal((3, 40, 24)) * np.exp(rng.uniform(-8, 3, (3, 1, 24)))
    W[1, :, 5] = 0.0                                          # an all-zero column
    codes, scales = orc.quantize_fp8(W)
    t = _e4m3_table()
    keys = np.array(sorted(t, key=lambda b: (t[b], b)))
    vals = np.array([t[b] for b in keys])
    for m, r, c in itertools.product(range(3), range(0, 40, 7), range(24)):
        x = W[m, r, c] / scales[m, c]
        d = np.abs(vals - x)
        best = np.flatnonzero(d == d.min())
        got = t[int(codes[m, r, c])]
        assert got in vals[best]
        if len(best) > 1 and vals[best[0]] != vals[best[-1]]:   # a genuine tie: even mantissa
            assert (int(codes[m, r, c]) & 1) == 0
    assert scales[1, 5] == 1.0 and np.all(codes[1, :, 5] & 0x7F == 0)


def test_scales_are_powers_of_two_and_cover_the_column():
    rng = np.random.default_rng(1)
    W = rng.standard_normal((2, 64, 32)) * 0.02
    codes, scales = orc.quantize_fp8(W)
    assert np.all(np.exp2(np.round(np.log2(scales))) == scales)
    amax = np.abs(W).max(axis=1)
    assert np.all(amax / scales <= 448.0) and np.all(amax / scales > 224.0)
    deq = orc.dequantize_fp8(codes, scales)
    rel = np.abs(deq - W) / np.maximum(np.abs(W), 1e-300)
    big = np.abs(W) >= 2.0 ** -6 * scales[:, None, :]        # normal range: 3 mantissa bits
    assert np.all(rel[big] <= 2.0 ** -4 + 1e-12)
    # dequantised values are bf16-exact
    assert np.array_equal(torch.tensor(deq).to(torch.bfloat16).double().numpy(), deq)
