"""GPU parity of the packed-sequence metadata (through the C ABI) against the CPU oracle:
bit for bit, integers throughout."""
import numpy as np
import pytest
import torch

from oracle import packed_oracle as po

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _positions(lengths):
    return np.concatenate([np.arange(L) for L in lengths]) if len(lengths) else np.zeros(0, np.int64)


def _check(pos, dtype, with_mask=True):
    import moe_expert_dispatch_stable_gb300 as moe
    meta = moe.moe_packed_metadata(torch.from_numpy(np.asarray(pos, dtype=np.int64)).to("cuda", dtype))
    torch.cuda.synchronize()
    cu, seq_id, n, mx = po.packed_metadata(pos)
    assert int(meta.n_seqs.item()) == n and int(meta.max_seqlen.item()) == mx
    assert np.array_equal(meta.cu_seqlens.cpu().numpy()[: n + 1], cu)
    assert np.array_equal(meta.seq_id.cpu().numpy(), seq_id)
    if with_mask:
        mask = moe.moe_packed_causal_mask(meta)
        torch.cuda.synchronize()
        assert np.array_equal(mask.cpu().numpy().astype(np.uint8), po.packed_causal_mask(seq_id))
    return meta


@pytest.mark.parametrize("dtype", [torch.int32, torch.int64])
def test_golden_and_two_sequences_of_2048(dtype):
    import json, os
    for case in json.load(open(os.path.join(os.path.dirname(__file__), "golden", "packed_hand_case.json")))["cases"]:
        _check(case["position_ids"], dtype)
    meta = _check(_positions([2048, 2048]), dtype)
    assert meta.cu_seqlens.cpu().tolist()[:3] == [0, 2048, 4096]


@pytest.mark.parametrize("seed", range(4))
def test_random_packings_across_chunks(seed):
    """Lengths 1..3000: tens of samples, several 4096-token chunks of the kernel, and
    mask rows whose length is not a multiple of 16."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(1, 3000, size=rng.integers(2, 12))
    _check(_positions(lengths), torch.int64 if seed % 2 else torch.int32, with_mask=seed < 2)


def test_row_kernel_mixed_chunks():
    """T a multiple of 16 (the row-wise mask kernel) with sample boundaries inside chunks."""
    lengths = [100, 1, 300, 2047, 48]
    assert sum(lengths) % 16 == 0
    _check(_positions(lengths), torch.int32)


@pytest.mark.parametrize("T", [1, 15, 16, 17, 4095, 4096, 4097])
def test_edge_sizes(T):
    _check(np.zeros(T, np.int64), torch.int32)            # every token its own sample
    _check(np.arange(T) + 5, torch.int64)                 # one sample, first position id not 0


def test_empty_batch_and_cache():
    import moe_expert_dispatch_stable_gb300 as moe
    meta = moe.moe_packed_metadata(torch.zeros(0, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert int(meta.n_seqs.item()) == 0 and int(meta.max_seqlen.item()) == 0 and meta.cu_seqlens.tolist() == [0]
    assert moe.moe_packed_causal_mask(meta).shape == (0, 0)
    pb = moe.PackedBatch(torch.from_numpy(_positions([3, 5, 2])).cuda())
    assert pb.host_sizes() == (3, 5)
    assert pb.cu_seqlens().tolist() == [0, 3, 8, 10]
    assert pb.causal_mask() is pb.causal_mask()             # built once, then reused
    # rebuilding into the same buffers
    again = moe.moe_packed_metadata(torch.from_numpy(_positions([4, 1, 5])).cuda(), out=pb.meta)
    torch.cuda.synchronize()
    assert again.cu_seqlens.data_ptr() == pb.meta.cu_seqlens.data_ptr()
    assert again.cu_seqlens.tolist()[:4] == [0, 4, 5, 10] and int(again.max_seqlen.item()) == 5


def test_long_batch():
    """About 180K tokens (44 chunks of the single-CTA kernel): metadata in full, no mask."""
    rng = np.random.default_rng(9)
    lengths = rng.integers(1, 9000, size=40)
    _check(_positions(lengths), torch.int64, with_mask=False)
