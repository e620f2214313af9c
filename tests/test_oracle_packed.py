"""Pins of the packed-sequence metadata oracle against things other than itself:
a hand-worked golden case, the two-sequences-of-2048 packing, packings built from
known lengths, and the mask against torch.block_diag of lower-triangular blocks."""
import json
import os

import numpy as np
import pytest

from oracle import packed_oracle as po

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "packed_hand_case.json")


def _cases():
    return json.load(open(GOLDEN))["cases"]


@pytest.mark.parametrize("case", _cases(), ids=["three_samples", "first_token_starts"])
def test_golden_hand_case(case):
    cu, seq_id, n, mx = po.packed_metadata(case["position_ids"])
    assert cu.tolist() == case["cu_seqlens"]
    assert seq_id.tolist() == case["seq_id"]
    assert n == case["n_seqs"] and mx == case["max_seqlen"]
    assert po.packed_causal_mask(seq_id).tolist() == case["mask"]


def test_two_sequences_of_2048():
    """The packing of the GPT-OSS-20B-shaped workload: two samples of 2048 tokens."""
    pos = np.concatenate([np.arange(2048), np.arange(2048)])
    cu, seq_id, n, mx = po.packed_metadata(pos)
    assert cu.tolist() == [0, 2048, 4096] and n == 2 and mx == 2048
    assert (seq_id[:2048] == 0).all() and (seq_id[2048:] == 1).all()


@pytest.mark.parametrize("seed", range(6))
def test_packings_from_known_lengths(seed):
    rng = np.random.default_rng(seed)
    lengths = rng.integers(1, 300, size=rng.integers(1, 40))
    pos = np.concatenate([np.arange(L) for L in lengths])
    cu, seq_id, n, mx = po.packed_metadata(pos)
    assert cu.tolist() == [0] + np.cumsum(lengths).tolist()
    assert n == lengths.size and mx == lengths.max()
    # token t lies in the sequence whose cumulative end first exceeds t
    t = np.arange(pos.size)
    assert np.array_equal(seq_id, np.searchsorted(np.cumsum(lengths), t, side="right"))


@pytest.mark.parametrize("seed", range(4))
def test_mask_against_block_diag(seed):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(100 + seed)
    lengths = rng.integers(1, 40, size=rng.integers(1, 8))
    pos = np.concatenate([np.arange(L) for L in lengths])
    _, seq_id, _, _ = po.packed_metadata(pos)
    ref = torch.block_diag(*[torch.ones(int(L), int(L), dtype=torch.uint8).tril() for L in lengths]).numpy()
    assert np.array_equal(po.packed_causal_mask(seq_id), ref)


def test_every_token_its_own_sequence_and_empty():
    cu, seq_id, n, mx = po.packed_metadata(np.zeros(7, dtype=np.int64))
    assert cu.tolist() == list(range(8)) and n == 7 and mx == 1
    assert np.array_equal(po.packed_causal_mask(seq_id), np.eye(7, dtype=np.uint8))
    cu, seq_id, n, mx = po.packed_metadata(np.zeros(0, dtype=np.int64))
    assert cu.tolist() == [0] and seq_id.size == 0 and n == 0 and mx == 0
    assert po.packed_causal_mask(seq_id).shape == (0, 0)


def test_planted_mistakes_fail_the_golden_case():
    """Two plausible slips, planted in copies of the oracle on the CPU, are caught."""
    c1, c2 = _cases()

    def starts_without_token0(position_ids):          # forgets that token 0 always starts
        return np.flatnonzero(np.asarray(position_ids) == 0)

    assert starts_without_token0(c2["position_ids"]).tolist() != c2["cu_seqlens"][:-1]
    _, seq_id, _, _ = po.packed_metadata(c1["position_ids"])
    transposed = po.packed_causal_mask(seq_id).T                     # j >= i instead of j <= i
    assert transposed.tolist() != c1["mask"]
