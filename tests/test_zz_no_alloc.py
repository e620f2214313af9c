"""moe_route_static: routing for callers that cannot allocate device memory.

Some callers of this library cannot call cudaMalloc: hosts whose device memory
belongs to another allocator or a fixed pool, and latency-critical loops where
an allocation might synchronise the device.  moe_route_static serves them: it
takes no workspace and keeps its scratch in a fixed device array inside the
library.  This test calls it through the C ABI (ctypes on the shared library)
twice in a row, with different sizes, and checks that each call's outputs are
bit-identical to those of moe_route, the entry point with a caller-provided
workspace (routing parity in this project is bit-exact).  It is collected last,
so that a run stopping at its first failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import moe_inputs as mi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from moe_expert_dispatch_stable_gb300 import binding
    lib = binding.load_library()
    vp = ctypes.c_void_p
    lib.moe_route_static.argtypes = [vp, ctypes.c_int32, vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                     ctypes.POINTER(binding.moe_routing), vp, vp]
    lib.moe_route_static.restype = ctypes.c_int32
    torch.cuda.set_device(0)
    return lib


def _static_route(lib, idx, w, E, dev_status):
    from moe_expert_dispatch_stable_gb300 import binding
    T, k = idx.shape
    out = binding.Routing.empty(T, k, E, idx.device)
    rt = out.c_struct()
    st = lib.moe_route_static(ctypes.c_void_p(idx.data_ptr()), idx.element_size(), ctypes.c_void_p(w.data_ptr()),
                              T, k, E, ctypes.byref(rt), ctypes.c_void_p(dev_status.data_ptr()),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out


def test_route_static_matches_route_on_consecutive_calls(lib):
    import moe_expert_dispatch_stable_gb300 as moe
    # consecutive calls of different sizes: the shared scratch keeps the previous call's contents
    for name, seed in [("gptoss120b_skew", 0), ("dsv3", 1), ("tiny", 2), ("gptoss120b_skew", 3)]:
        cfg = mi.CONFIGS[name]
        idx_np, w_np = mi.make_routing(cfg, seed)
        idx = torch.from_numpy(idx_np).cuda()
        w = torch.from_numpy(w_np).cuda()
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        st, got = _static_route(lib, idx, w, cfg.E, status)
        assert st == 0, lib.moe_status_string(st)
        ref = moe.moe_route(idx, w, cfg.E)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for field in ("perm", "inv_perm", "counts", "offsets", "tile_offsets"):
            assert torch.equal(getattr(got, field), getattr(ref, field)), (name, field)
        assert torch.equal(got.w_sorted.view(torch.int32), ref.w_sorted.view(torch.int32)), name


def test_route_static_rejects_sizes_beyond_its_scratch(lib):
    # E = 1024 and 64 chunks of 1024 slots need 256 KiB + 256 B of scratch: refused before any launch
    T, k, E = 16384, 4, 1024
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    st, _ = _static_route(lib, idx, w, E, status)
    assert st == 4                                          # MOE_ERR_WORKSPACE
    # one chunk fewer fits
    st, _ = _static_route(lib, idx[: 63 * 256], w[: 63 * 256], E, status)
    torch.cuda.synchronize()
    assert st == 0 and int(status.item()) == 0
