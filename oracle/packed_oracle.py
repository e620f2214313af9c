"""CPU oracle for packed-sequence metadata -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
import this module.  It shares no code with the CUDA path and imports nothing
from it.

Source: the "Unsloth and NVIDIA" blog post (d9249.github.io write-up of
Unsloth x NVIDIA's training speed-ups), section "core idea / structure / how
it works", first improvement (packed-sequence metadata caching).  Several
short samples are concatenated into one long token stream; the model still
needs each original sequence's length, the cumulative offsets (cu_seqlens),
the longest length and the attention structure, and these are the same for
every layer of one packed batch, so they are built once per batch and reused
instead of being rebuilt (with device-to-host copies) in every layer.

The pages do not say how a packed batch is described.  Read here in the usual
way for packed training: per-token position ids that restart at 0 at the
first token of every sample.  A sequence starts at token 0 and at every token
whose position id is 0.  The attention structure is the block-diagonal causal
mask: token i attends to token j iff both lie in the same sequence and j <= i.

Plain numpy on int64; every function is its definition written out.
Parity pins: tests/test_oracle_packed.py (a hand-worked golden case, the
two-sequences-of-2048 packing, the mask against torch.block_diag of
lower-triangular blocks, packings generated from known lengths).  No numeric
example is printed on the pages.
"""
from __future__ import annotations

import numpy as np


def sequence_starts(position_ids):
    """Token indices where a sequence starts: 0, and every t with position_ids[t] == 0."""
    pos = np.asarray(position_ids).reshape(-1).astype(np.int64)
    start = pos == 0
    if start.size:
        start[0] = True
    return np.flatnonzero(start).astype(np.int64)


def packed_metadata(position_ids):
    """(cu_seqlens [n+1], seq_id [T], n_seqs, max_seqlen) of a packed batch.

    cu_seqlens[s] is the first token of sequence s and cu_seqlens[n] = T;
    seq_id[t] is the sequence token t belongs to; max_seqlen is the longest
    sequence (0 for an empty batch).
    """
    T = int(np.asarray(position_ids).size)
    starts = sequence_starts(position_ids)
    cu = np.append(starts, T).astype(np.int64)
    lengths = np.diff(cu)
    n = int(starts.size)
    seq_id = np.repeat(np.arange(n, dtype=np.int64), lengths)
    max_seqlen = int(lengths.max()) if n else 0
    return cu, seq_id, n, max_seqlen


def packed_causal_mask(seq_id):
    """mask[i, j] = 1 iff tokens i and j lie in the same sequence and j <= i (uint8)."""
    s = np.asarray(seq_id).reshape(-1).astype(np.int64)
    T = s.size
    same = s[:, None] == s[None, :]
    causal = np.arange(T)[None, :] <= np.arange(T)[:, None]
    return (same & causal).astype(np.uint8)
