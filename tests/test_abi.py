"""The C-ABI library builds, loads and exports every symbol its header declares;
host-side argument checks return their status codes without a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


def _declared_symbols():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        names.update(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text, flags=re.M))
    return names


@pytest.fixture(scope="module")
def lib():
    from moe_expert_dispatch_stable_gb300 import build
    path = build.build()
    from moe_expert_dispatch_stable_gb300 import binding
    return binding.load_library(path)


def test_header_declares_the_three_operations():
    names = _declared_symbols()
    assert {"moe_route", "moe_lora_fwd", "moe_lora_bwd"} <= names
    assert len(names) >= 9


def test_library_exports_every_declared_symbol(lib):
    for name in sorted(_declared_symbols()):
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_abi_version_and_status_strings(lib):
    assert lib.moe_abi_version() == 7
    for code in range(0, 7):
        assert lib.moe_status_string(code)


def test_size_queries_and_dim_checks(lib):
    from moe_expert_dispatch_stable_gb300 import binding as b
    n = ctypes.c_size_t()
    assert lib.moe_route_workspace_size(4096, 4, 32, ctypes.byref(n)) == 0 and n.value > 0
    assert lib.moe_route_workspace_size(4096, 4, 2048, ctypes.byref(n)) == 2       # E > 1024
    assert lib.moe_route_workspace_size(4096, 5, 4, ctypes.byref(n)) == 2          # k > E
    assert lib.moe_route_workspace_size(-1, 1, 4, ctypes.byref(n)) == 2
    assert lib.moe_route_workspace_size(4096, 4, 32, None) == 1
    ok = b.Dims(T=4096, H=2880, I=2880, E=32, k=4, r=16, scale=2.0)
    saved, ws = b.moe_lora_fwd_sizes(ok)
    N = 4096 * 4
    assert saved >= N * 2880 * 2 + N * 5760 * 2 + N * 2880 * 2 + 2 * N * 16 * 2
    assert ws == 0                                          # the forward keeps everything in `saved`
    assert saved >= N * (2880 * 2 + 5760 * 2 + 2880 * 2 + 2 * 16 * 2 + 2880 * 2)
    # dO, G_s, dGU, Gg_s and the bf16 dX rows of the routed slots
    bws = b.moe_lora_bwd_workspace_size(ok)
    assert N * (2880 * 2 + 16 * 2 + 5760 * 2 + 16 * 2 + 2880 * 2) <= bws <= N * (2880 * 2 + 16 * 2 + 5760 * 2 + 16 * 2 + 2880 * 2) + 5 * 256
    offs, rp = b.moe_lora_saved_layout(ok)
    assert rp == 16 and offs[0] == 0 and all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    assert b.moe_lora_saved_layout(b.Dims(64, 128, 256, 8, 2, 8, 2.0))[1] == 16
    assert b.moe_lora_saved_layout(b.Dims(64, 128, 256, 8, 2, 32, 2.0))[1] == 32
    for bad in [dict(H=100), dict(I=96 + 1), dict(r=0), dict(r=65), dict(k=40), dict(E=0)]:
        d = b.Dims(**{**ok.__dict__, **bad})
        with pytest.raises(b.MoEError):
            b.moe_lora_fwd_sizes(d)


def test_null_and_misaligned_arguments_rejected_before_launch(lib):
    from moe_expert_dispatch_stable_gb300 import binding as b
    rt = b.moe_routing(16, 16, 16, 16, 16, 16)
    # NULL topk_idx with T > 0
    assert lib.moe_route(None, 4, ctypes.c_void_p(16), 8, 2, 4, ctypes.byref(rt), ctypes.c_void_p(16), 1 << 20,
                         ctypes.c_void_p(16), None) == 1
    # a NULL routing output
    rt_bad = b.moe_routing(16, 0, 16, 16, 16, 16)
    assert lib.moe_route(ctypes.c_void_p(16), 4, ctypes.c_void_p(16), 8, 2, 4, ctypes.byref(rt_bad),
                         ctypes.c_void_p(16), 1 << 20, ctypes.c_void_p(16), None) == 1
    # misaligned topk_idx
    assert lib.moe_route(ctypes.c_void_p(18), 4, ctypes.c_void_p(16), 8, 2, 4, ctypes.byref(rt),
                         ctypes.c_void_p(16), 1 << 20, ctypes.c_void_p(16), None) == 3
    # workspace too small
    assert lib.moe_route(ctypes.c_void_p(16), 4, ctypes.c_void_p(16), 8, 2, 4, ctypes.byref(rt),
                         ctypes.c_void_p(16), 4, ctypes.c_void_p(16), None) == 4
    # bad index width
    assert lib.moe_route(ctypes.c_void_p(16), 2, ctypes.c_void_p(16), 8, 2, 4, ctypes.byref(rt),
                         ctypes.c_void_p(16), 1 << 20, ctypes.c_void_p(16), None) == 2
    d = b.Dims(8, 64, 64, 4, 2, 4, 2.0).c_struct()
    # weights 16-byte aligned, activation buffers (x, y, dy, dx, saved, workspace) 32-byte aligned
    w16, a32, a16 = ctypes.c_void_p(16), ctypes.c_void_p(32), ctypes.c_void_p(48)
    wts = [w16] * 6
    assert lib.moe_lora_fwd(ctypes.byref(d), ctypes.byref(rt), a32, *wts, None, a32, 1 << 30,
                            a32, 1 << 30, w16, None) == 1
    assert lib.moe_lora_fwd(ctypes.byref(d), ctypes.byref(rt), a32, *wts, a32, a32, 1,
                            a32, 1 << 30, w16, None) == 4
    # x, y, saved or workspace only 16-byte aligned
    for bad in range(4):
        acts = [a16 if i == bad else a32 for i in range(4)]
        assert lib.moe_lora_fwd(ctypes.byref(d), ctypes.byref(rt), acts[0], *wts, acts[1], acts[2], 1 << 30,
                                acts[3], 1 << 30, w16, None) == 3
    assert lib.moe_lora_bwd(ctypes.byref(d), ctypes.byref(rt), a32, *wts, a32, 1 << 30,
                            ctypes.c_void_p(24), *[w16] * 4, None, a32, 1 << 30, w16, None) == 3
    assert lib.moe_lora_bwd(ctypes.byref(d), ctypes.byref(rt), a32, *wts, a32, 1 << 30,
                            a16, *[w16] * 4, None, a32, 1 << 30, w16, None) == 3
    # regather: NULL x, 16-byte aligned saved, saved buffer too small
    assert lib.moe_lora_saved_regather(ctypes.byref(d), ctypes.byref(rt), None, a32, 1 << 30, None) == 1
    assert lib.moe_lora_saved_regather(ctypes.byref(d), ctypes.byref(rt), a32, a16, 1 << 30, None) == 3
    assert lib.moe_lora_saved_regather(ctypes.byref(d), ctypes.byref(rt), a32, a32, 16, None) == 4
    # rebuild of h: NULL / 16-byte aligned / too small saved buffer
    assert lib.moe_lora_saved_rebuild_h(ctypes.byref(d), None, 1 << 30, None) == 1
    assert lib.moe_lora_saved_rebuild_h(ctypes.byref(d), a16, 1 << 30, None) == 3
    assert lib.moe_lora_saved_rebuild_h(ctypes.byref(d), a32, 16, None) == 4
    # misaligned d_topk_w
    assert lib.moe_lora_bwd(ctypes.byref(d), ctypes.byref(rt), a32, *wts, a32, 1 << 30,
                            a32, *[w16] * 4, ctypes.c_void_p(20), a32, 1 << 30, w16, None) == 3
    # router: bad sizes, NULL outputs, misaligned logits
    assert lib.moe_router_topk(ctypes.c_void_p(16), 8, 4, 5, ctypes.c_void_p(16), ctypes.c_void_p(16), None) == 2
    assert lib.moe_router_topk(ctypes.c_void_p(16), 8, 2048, 2, ctypes.c_void_p(16), ctypes.c_void_p(16), None) == 2
    assert lib.moe_router_topk(ctypes.c_void_p(16), 8, 4, 2, None, ctypes.c_void_p(16), None) == 1
    assert lib.moe_router_topk(ctypes.c_void_p(20), 8, 4, 2, ctypes.c_void_p(16), ctypes.c_void_p(16), None) == 3
    assert lib.moe_router_bwd(ctypes.c_void_p(16), ctypes.c_void_p(16), None, 8, 4, 2, ctypes.c_void_p(16),
                              None) == 1


def test_fp8_entry_points_host_checks(lib):
    from moe_expert_dispatch_stable_gb300 import binding as b
    v = ctypes.c_void_p
    # quantiser: negative sizes, NULL buffers with a non-empty tensor, misalignment
    assert lib.moe_quantize_fp8(v(16), -1, 4, 64, v(16), v(16), None) == 2
    assert lib.moe_quantize_fp8(None, 2, 4, 64, v(16), v(16), None) == 1
    assert lib.moe_quantize_fp8(v(16), 2, 4, 64, v(24), v(16), None) == 3
    rt = b.moe_routing(16, 16, 16, 16, 16, 16)
    d = b.Dims(8, 64, 64, 4, 2, 4, 2.0).c_struct()
    w16, a32 = v(16), v(32)

    def fwd(s_gu, s_d):
        return lib.moe_lora_fwd_fp8(ctypes.byref(d), ctypes.byref(rt), a32, w16, s_gu, w16, w16, w16, s_d, w16, w16,
                                    a32, a32, 1 << 30, a32, 1 << 30, w16, None)

    def bwd(s_gu, s_d):
        return lib.moe_lora_bwd_fp8(ctypes.byref(d), ctypes.byref(rt), a32, w16, s_gu, w16, w16, w16, s_d, w16, w16,
                                    a32, 1 << 30, a32, w16, w16, w16, w16, None, a32, 1 << 30, w16, None)

    # the column scales are required and 16-byte aligned
    for call in (fwd, bwd):
        assert call(None, w16) == 1 and call(w16, None) == 1
        assert call(v(20), w16) == 3 and call(w16, v(20)) == 3


def test_nf4_entry_points_host_checks(lib):
    from moe_expert_dispatch_stable_gb300 import binding as b
    v = ctypes.c_void_p
    # quantiser: rows of a multiple of 64 elements, NULL buffers with a non-empty tensor, misalignment
    assert lib.moe_quantize_nf4(v(16), 2, 4, 96, v(16), v(16), None) == 2
    assert lib.moe_quantize_nf4(v(16), -1, 4, 64, v(16), v(16), None) == 2
    assert lib.moe_quantize_nf4(None, 2, 4, 64, v(16), v(16), None) == 1
    assert lib.moe_quantize_nf4(v(16), 2, 4, 64, v(16), v(24), None) == 3
    assert lib.moe_quantize_nf4(None, 0, 4, 64, None, None, None) == 0        # empty: nothing to do
    assert lib.moe_nf4_codebook(None) == 1
    rt = b.moe_routing(16, 16, 16, 16, 16, 16)
    d = b.Dims(8, 64, 64, 4, 2, 4, 2.0).c_struct()
    w16, a32 = v(16), v(32)

    def fwd(m_gu, m_d):
        return lib.moe_lora_fwd_nf4(ctypes.byref(d), ctypes.byref(rt), a32, w16, m_gu, w16, w16, w16, m_d, w16, w16,
                                    a32, a32, 1 << 30, a32, 1 << 30, w16, None)

    def bwd(m_gu, m_d):
        return lib.moe_lora_bwd_nf4(ctypes.byref(d), ctypes.byref(rt), a32, w16, m_gu, w16, w16, w16, m_d, w16, w16,
                                    a32, 1 << 30, a32, w16, w16, w16, w16, None, a32, 1 << 30, w16, None)

    # the block scales are required and 16-byte aligned
    for call in (fwd, bwd):
        assert call(None, w16) == 1 and call(w16, None) == 1
        assert call(v(20), w16) == 3 and call(w16, v(20)) == 3


def test_nf4_codebook_equals_the_oracle_bit_for_bit(lib):
    """The library computes its 16 NF4 values on the host from their definition (inverse
    normal CDF by bisection on erfc); the oracle takes scipy's inverse CDF.  Both round to
    float32, and the tables agree bit for bit."""
    import numpy as np

    from moe_expert_dispatch_stable_gb300 import binding as b
    from oracle import nf4_oracle as nf
    got = np.array(b.moe_nf4_codebook(), dtype=np.float32)
    np.testing.assert_array_equal(got.view(np.uint32), nf.nf4_codebook().view(np.uint32))


def test_timing_diagnostics_host_side(lib):
    """Timing diagnostics without a launch: NULL outputs, and an index past the last name."""
    name = ctypes.create_string_buffer(64)
    ms, n = ctypes.c_double(), ctypes.c_int32()
    assert lib.moe_timing_enable(1) == 0           # clears the record
    assert lib.moe_timing_read(0, None, 64, ctypes.byref(ms), ctypes.byref(n)) == 1
    assert lib.moe_timing_read(0, name, 0, ctypes.byref(ms), ctypes.byref(n)) == 1
    assert lib.moe_timing_read(0, name, 64, ctypes.byref(ms), ctypes.byref(n)) == 2
    assert lib.moe_timing_read(-1, name, 64, ctypes.byref(ms), ctypes.byref(n)) == 2
    assert lib.moe_timing_enable(0) == 0
    assert lib.moe_launch_count() >= 0


def test_packed_metadata_host_checks(lib):
    v = ctypes.c_void_p
    # T out of range, bad position width
    assert lib.moe_packed_metadata(v(16), 4, -1, v(16), v(16), v(16), v(16), None) == 2
    assert lib.moe_packed_metadata(v(16), 4, (1 << 30) + 1, v(16), v(16), v(16), v(16), None) == 2
    assert lib.moe_packed_metadata(v(16), 2, 8, v(16), v(16), v(16), v(16), None) == 2
    # NULL outputs; NULL position ids with T > 0
    assert lib.moe_packed_metadata(v(16), 4, 8, None, v(16), v(16), v(16), None) == 1
    assert lib.moe_packed_metadata(None, 4, 8, v(16), v(16), v(16), v(16), None) == 1
    # int64 position ids aligned to 4 only; a misaligned int32 output
    assert lib.moe_packed_metadata(v(20), 8, 8, v(16), v(16), v(16), v(16), None) == 3
    assert lib.moe_packed_metadata(v(16), 4, 8, v(18), v(16), v(16), v(16), None) == 3
    # the mask: NULL, 16-byte alignment, T out of range
    assert lib.moe_packed_causal_mask(v(16), v(16), 8, None, None) == 1
    assert lib.moe_packed_causal_mask(v(16), v(16), 8, v(24), None) == 3
    assert lib.moe_packed_causal_mask(v(16), v(16), -3, v(16), None) == 2


def test_binding_fails_loudly_without_library(tmp_path):
    from moe_expert_dispatch_stable_gb300 import binding as b
    with pytest.raises(b.MoEError):
        b.load_library(str(tmp_path / "missing.so"))
    with pytest.raises(b.MoEError):
        with b.using_library(str(tmp_path / "missing.so")):
            pass


def test_debug_build_loads_and_exports_the_same_symbols():
    """The debug build (MOE_DEBUG=1: routing indices checked, MOE_DEV_BAD_INDEX) builds,
    loads and exports every declared symbol, with the same ABI version."""
    from moe_expert_dispatch_stable_gb300 import binding as b, build
    path = build.build(debug=True)
    assert path == b.LIB_DEBUG_PATH
    dbg = b.load_library(path)
    assert dbg.moe_abi_version() == b.ABI_VERSION
    for name in sorted(_declared_symbols()):
        assert hasattr(dbg, name), f"{name} missing from the debug build"
    with b.using_library(path) as lib:
        assert lib is dbg and b.load_library() is dbg
    assert b.load_library() is not dbg


def _header_arity():
    """Number of parameters of every MOE_API function in include/ (void -> 0)."""
    out = {}
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(([^)]*)\)\s*;", text):
            params = [p for p in m.group(2).split(",") if p.strip()]
            out[m.group(1)] = 0 if params == ["void"] or [p.strip() for p in params] == ["void"] else len(params)
    return out


def test_binding_argtypes_match_header_arity(lib):
    from moe_expert_dispatch_stable_gb300 import binding as b
    arity = _header_arity()
    assert len(arity) >= 18
    for name in b.EXPORTED:                     # every function the binding wraps
        argtypes = getattr(lib, name).argtypes
        n = arity[name]
        if argtypes is None:
            assert n == 0, f"{name}: no argtypes set but the header declares {n} parameters"
        else:
            assert len(argtypes) == n, f"{name}: binding declares {len(argtypes)} arguments, header {n}"


def test_forced_timeout_hook_checks_its_limit(lib):
    """The failure-path hook takes a wait limit in [1 us, 2 s] and disarms on a negative index;
    checked on the host, nothing is launched."""
    assert lib.moe_diag_force_timeout(0, 999) == 2
    assert lib.moe_diag_force_timeout(0, 2_000_000_001) == 2
    assert lib.moe_diag_force_timeout(-1, 0) == 0
    assert lib.moe_diag_force_timeout(3, 1_000_000) == 0
    assert lib.moe_diag_force_timeout(-1, 0) == 0


def test_layer_rejects_h_from_gu_with_quantised_weights():
    """The h-from-GU forward exists for bf16 weights only; a layer over quantised weights
    refuses the flag before allocating anything."""
    from moe_expert_dispatch_stable_gb300 import binding as b
    d = b.Dims(8, 64, 64, 4, 2, 4, 2.0)
    for key in ("Wq_gu", "W4_gu"):
        with pytest.raises(b.MoEError):
            b.MoELoRALayer(d, {key: None}, device="cpu", h_from_gu=True)
