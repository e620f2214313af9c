"""The gather of the permuted rows (x_perm[p] = x[perm[p] / k]; one warp per sorted row
and 4 KB chunk of it, 32-byte accesses) bit for bit at its edges: rows narrower than one
chunk, widths with a ragged last chunk, odd row counts, one token, and the widest
workload row (7168 columns)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("T,k,E,H", [(1, 1, 2, 64), (1, 2, 4, 64), (3, 1, 2, 128), (5, 3, 7, 192), (257, 2, 8, 320),
                                     (1001, 3, 16, 2880), (4096, 4, 32, 2880), (333, 8, 64, 7168)])
def test_gather_rows_bit_exact(T, k, E, H):
    import moe_expert_dispatch_stable_gb300 as moe
    rng = np.random.default_rng(T * 7 + H)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int64)
    w = rng.random((T, k)).astype(np.float32)
    x = torch.randn((T, H), dtype=torch.float32).to(torch.bfloat16).cuda()
    d = moe.Dims(T, H, 64, E, k, 4, 2.0)
    rt = moe.moe_route(torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), E)
    saved_bytes, _ = moe.moe_lora_fwd_sizes(d)
    saved = torch.full((saved_bytes,), 0x5A, dtype=torch.uint8, device="cuda")
    moe.moe_lora_saved_regather(d, rt, x, saved)
    torch.cuda.synchronize()
    offs, _ = moe.moe_lora_saved_layout(d)
    N = T * k
    xp = saved[offs[0]:offs[0] + N * H * 2].view(torch.bfloat16).view(N, H)
    perm = rt.perm.long()
    assert torch.equal(xp, x[perm // k])
    # nothing past the section was written
    assert torch.all(saved[offs[0] + N * H * 2:offs[1]] == 0x5A)
