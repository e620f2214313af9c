"""Thin Python binding of the MoE-LoRA C ABI (``include/moe_lora.h``).

Argument marshalling only: torch tensors are checked for device, dtype,
contiguity and shape, and their data pointers, sizes and the current CUDA
stream are handed to the C functions of the same names.  Every step of the
layer runs in the library's kernels; there is no fallback of any kind -- if
the shared library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_lora_gb300.so")
# the debug build: indices read from routing buffers are checked (MOE_DEV_BAD_INDEX)
LIB_DEBUG_PATH = os.path.join(_PKG, "libmoe_lora_gb300_debug.so")

MOE_OK = 0
MOE_DEV_BAD_EXPERT_ID = 1
MOE_DEV_TIMEOUT = 2
MOE_DEV_BAD_INDEX = 4
TILE_M = 128


class MoEError(RuntimeError):
    pass


class moe_dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("r", ctypes.c_int32),
                ("scale", ctypes.c_float)]


class moe_routing(ctypes.Structure):
    _fields_ = [("perm", ctypes.c_void_p), ("inv_perm", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("tile_offsets", ctypes.c_void_p), ("w_sorted", ctypes.c_void_p)]


EXPORTED = ("moe_abi_version", "moe_status_string", "moe_launch_count", "moe_route_workspace_size", "moe_route",
            "moe_lora_fwd_sizes", "moe_lora_saved_layout", "moe_lora_saved_regather", "moe_lora_saved_rebuild_h", "moe_lora_fwd", "moe_lora_fwd_h_from_gu",
            "moe_lora_bwd_workspace_size", "moe_lora_bwd", "moe_timing_enable", "moe_timing_read",
            "moe_router_topk", "moe_router_bwd", "moe_quantize_fp8", "moe_lora_fwd_fp8", "moe_lora_bwd_fp8",
            "moe_quantize_nf4", "moe_nf4_codebook", "moe_lora_fwd_nf4", "moe_lora_bwd_nf4",
            "moe_packed_metadata", "moe_packed_causal_mask", "moe_diag_force_timeout")
ABI_VERSION = 7

_libs: dict = {}
_default_path = LIB_PATH


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built).  Without `path`: the library
    the binding's calls currently go to (the release build unless `using_library` says so)."""
    path = path or _default_path
    if path in _libs:
        return _libs[path]
    if not os.path.exists(path):
        raise MoEError(f"MoE-LoRA CUDA library not built: {path} is missing "
                       "(run moe_expert_dispatch_stable_gb300.build.build())")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    P = ctypes.POINTER
    lib.moe_abi_version.restype = i32
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_status_string.argtypes = [i32]
    lib.moe_route_workspace_size.argtypes = [i64, i32, i32, P(sz)]
    lib.moe_route.argtypes = [vp, i32, vp, i64, i32, i32, P(moe_routing), vp, sz, vp, vp]
    lib.moe_lora_fwd_sizes.argtypes = [P(moe_dims), P(sz), P(sz)]
    lib.moe_lora_saved_layout.argtypes = [P(moe_dims), P(sz), P(i32)]
    lib.moe_lora_saved_regather.argtypes = [P(moe_dims), P(moe_routing), vp, vp, sz, vp]
    lib.moe_lora_saved_rebuild_h.argtypes = [P(moe_dims), vp, sz, vp]
    lib.moe_lora_fwd.argtypes = [P(moe_dims), P(moe_routing)] + [vp] * 8 + [vp, sz, vp, sz, vp, vp]
    lib.moe_lora_fwd_h_from_gu.argtypes = lib.moe_lora_fwd.argtypes
    lib.moe_lora_bwd_workspace_size.argtypes = [P(moe_dims), P(sz)]
    lib.moe_lora_bwd.argtypes = [P(moe_dims), P(moe_routing)] + [vp] * 7 + [vp, sz] + [vp] * 6 + [vp, sz, vp, vp]
    lib.moe_router_topk.argtypes = [vp, i64, i32, i32, vp, vp, vp]
    lib.moe_quantize_fp8.argtypes = [vp, i64, i64, i32, vp, vp, vp]
    lib.moe_lora_fwd_fp8.argtypes = [P(moe_dims), P(moe_routing)] + [vp] * 10 + [vp, sz, vp, sz, vp, vp]
    lib.moe_lora_bwd_fp8.argtypes = [P(moe_dims), P(moe_routing)] + [vp] * 10 + [sz] + [vp] * 6 + [vp, sz, vp, vp]
    lib.moe_quantize_nf4.argtypes = lib.moe_quantize_fp8.argtypes
    lib.moe_nf4_codebook.argtypes = [P(ctypes.c_float)]
    lib.moe_lora_fwd_nf4.argtypes = lib.moe_lora_fwd_fp8.argtypes
    lib.moe_lora_bwd_nf4.argtypes = lib.moe_lora_bwd_fp8.argtypes
    lib.moe_router_bwd.argtypes = [vp, vp, vp, i64, i32, i32, vp, vp]
    lib.moe_packed_metadata.argtypes = [vp, i32, i64, vp, vp, vp, vp, vp]
    lib.moe_packed_causal_mask.argtypes = [vp, vp, i64, vp, vp]
    lib.moe_launch_count.restype = ctypes.c_uint64
    lib.moe_timing_enable.argtypes = [i32]
    lib.moe_timing_read.argtypes = [i32, ctypes.c_char_p, sz, P(ctypes.c_double), P(i32)]
    lib.moe_diag_force_timeout.argtypes = [i32, ctypes.c_uint64]
    for name in EXPORTED[3:]:
        getattr(lib, name).restype = i32
    if lib.moe_abi_version() != ABI_VERSION:
        raise MoEError("MoE-LoRA library ABI version mismatch")
    _libs[path] = lib
    return lib


@contextlib.contextmanager
def using_library(path: str):
    """Send the binding's calls to the library at `path` (e.g. LIB_DEBUG_PATH, the build
    that checks routing indices) inside the block; process-wide."""
    global _default_path
    old = _default_path
    lib = load_library(path)
    _default_path = path
    try:
        yield lib
    finally:
        _default_path = old


def _check(status: int):
    if status != MOE_OK:
        msg = load_library().moe_status_string(status).decode()
        raise MoEError(f"MoE-LoRA call failed with status {status}: {msg}")


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise MoEError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise MoEError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise MoEError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise MoEError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


@dataclass
class Routing:
    perm: torch.Tensor
    inv_perm: torch.Tensor
    counts: torch.Tensor
    offsets: torch.Tensor
    tile_offsets: torch.Tensor
    w_sorted: torch.Tensor

    def c_struct(self) -> moe_routing:
        return moe_routing(self.perm.data_ptr(), self.inv_perm.data_ptr(), self.counts.data_ptr(),
                           self.offsets.data_ptr(), self.tile_offsets.data_ptr(), self.w_sorted.data_ptr())

    @staticmethod
    def empty(T: int, k: int, E: int, device) -> "Routing":
        N = T * k
        i32 = dict(dtype=torch.int32, device=device)
        return Routing(torch.empty(max(N, 4), **i32)[:N], torch.empty(max(N, 4), **i32)[:N],
                       torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(E + 1, **i32),
                       torch.empty(max(N, 4), dtype=torch.float32, device=device)[:N])


@dataclass(frozen=True)
class Dims:
    T: int
    H: int
    I: int
    E: int
    k: int
    r: int
    scale: float

    def c_struct(self) -> moe_dims:
        return moe_dims(self.T, self.H, self.I, self.E, self.k, self.r, self.scale)


def moe_route_workspace_size(T: int, k: int, E: int) -> int:
    n = ctypes.c_size_t()
    _check(load_library().moe_route_workspace_size(T, k, E, ctypes.byref(n)))
    return n.value


def moe_route(topk_idx: torch.Tensor, topk_w: torch.Tensor, E: int, out: Routing | None = None,
              workspace: torch.Tensor | None = None, dev_status: torch.Tensor | None = None,
              stream=None) -> Routing:
    """Group the T*k routed slots by expert (see moe_route in moe_lora.h)."""
    lib = load_library()
    if topk_idx.dtype not in (torch.int32, torch.int64):
        raise MoEError("topk_idx must be int32 or int64")
    _need(topk_idx, "topk_idx", topk_idx.dtype)
    if topk_idx.dim() != 2:
        raise MoEError("topk_idx must be [T, k]")
    T, k = topk_idx.shape
    _need(topk_w, "topk_w", torch.float32, (T, k))
    dev = topk_idx.device
    if out is None:
        out = Routing.empty(T, k, E, dev)
    if workspace is None:
        workspace = torch.empty(moe_route_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    rt = out.c_struct()
    _check(lib.moe_route(_ptr(topk_idx), topk_idx.element_size(), _ptr(topk_w), T, k, E, ctypes.byref(rt),
                         _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream(stream)))
    return out


def moe_lora_fwd_sizes(d: Dims):
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load_library().moe_lora_fwd_sizes(ctypes.byref(d.c_struct()), ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def moe_lora_saved_layout(d: Dims):
    offs = (ctypes.c_size_t * 6)()
    rp = ctypes.c_int32()
    _check(load_library().moe_lora_saved_layout(ctypes.byref(d.c_struct()), offs, ctypes.byref(rp)))
    return list(offs), rp.value


def moe_lora_saved_regather(d: Dims, rt: "Routing", x, saved, stream=None):
    """Re-create the x_perm section of `saved` from the layer input x (the forward's gather)."""
    _need(x, "x", torch.bfloat16, (d.T, d.H))
    dd, rr = d.c_struct(), rt.c_struct()
    _check(load_library().moe_lora_saved_regather(ctypes.byref(dd), ctypes.byref(rr), _ptr(x), _ptr(saved),
                                                  saved.numel() * saved.element_size(), _stream(stream)))


def moe_lora_saved_rebuild_h(d: Dims, saved, stream=None):
    """Re-create the h section of `saved` from its GU section (bit-identical to the forward's h)."""
    dd = d.c_struct()
    _check(load_library().moe_lora_saved_rebuild_h(ctypes.byref(dd), _ptr(saved), saved.numel() * saved.element_size(),
                                                   _stream(stream)))


def moe_lora_bwd_workspace_size(d: Dims) -> int:
    n = ctypes.c_size_t()
    _check(load_library().moe_lora_bwd_workspace_size(ctypes.byref(d.c_struct()), ctypes.byref(n)))
    return n.value


def _check_weights(d: Dims, W_gu, A_gu, B_gu, W_d, A_d, B_d):
    bf = torch.bfloat16
    _need(W_gu, "W_gu", bf, (d.E, d.H, 2 * d.I))
    _need(A_gu, "A_gu", bf, (d.E, d.r, d.H))
    _need(B_gu, "B_gu", bf, (d.E, d.r, 2 * d.I))
    _need(W_d, "W_d", bf, (d.E, d.I, d.H))
    _need(A_d, "A_d", bf, (d.E, d.r, d.I))
    _need(B_d, "B_d", bf, (d.E, d.r, d.H))


def moe_lora_fwd(d: Dims, rt: Routing, x, W_gu, A_gu, B_gu, W_d, A_d, B_d, y=None, saved=None,
                 workspace=None, dev_status=None, stream=None, h_from_gu=False):
    """Forward of the layer; returns (y, saved).  h_from_gu: form h from the stored bf16
    GU (moe_lora_fwd_h_from_gu), so that moe_lora_saved_rebuild_h can re-create it."""
    lib = load_library()
    _need(x, "x", torch.bfloat16, (d.T, d.H))
    _check_weights(d, W_gu, A_gu, B_gu, W_d, A_d, B_d)
    dev = x.device
    saved_b, ws_b = moe_lora_fwd_sizes(d)
    if y is None:
        y = torch.empty((d.T, d.H), dtype=torch.bfloat16, device=dev)
    if saved is None:
        saved = torch.empty(max(saved_b, 16), dtype=torch.uint8, device=dev)
    if workspace is None:
        workspace = torch.empty(max(ws_b, 16), dtype=torch.uint8, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    _need(y, "y", torch.bfloat16, (d.T, d.H))
    dd, rr = d.c_struct(), rt.c_struct()
    fn = lib.moe_lora_fwd_h_from_gu if h_from_gu else lib.moe_lora_fwd
    _check(fn(ctypes.byref(dd), ctypes.byref(rr), _ptr(x), _ptr(W_gu), _ptr(A_gu), _ptr(B_gu),
              _ptr(W_d), _ptr(A_d), _ptr(B_d), _ptr(y), _ptr(saved), saved.numel(),
              _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream(stream)))
    return y, saved


def moe_lora_bwd(d: Dims, rt: Routing, dy, W_gu, A_gu, B_gu, W_d, A_d, B_d, saved, dx=None, grads=None,
                 workspace=None, dev_status=None, stream=None, d_topk_w=None):
    """Backward of the layer; returns (dx, dA_gu, dB_gu, dA_d, dB_d).  When d_topk_w
    (a [T, k] float32 CUDA tensor) is given it receives dL/d topk_w."""
    lib = load_library()
    _need(dy, "dy", torch.bfloat16, (d.T, d.H))
    _check_weights(d, W_gu, A_gu, B_gu, W_d, A_d, B_d)
    dev = dy.device
    if dx is None:
        dx = torch.empty((d.T, d.H), dtype=torch.bfloat16, device=dev)
    if grads is None:
        grads = (torch.empty_like(A_gu), torch.empty_like(B_gu), torch.empty_like(A_d), torch.empty_like(B_d))
    if workspace is None:
        workspace = torch.empty(max(moe_lora_bwd_workspace_size(d), 16), dtype=torch.uint8, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    dA_gu, dB_gu, dA_d, dB_d = grads
    if d_topk_w is not None:
        _need(d_topk_w, "d_topk_w", torch.float32, (d.T, d.k))
    dd, rr = d.c_struct(), rt.c_struct()
    _check(lib.moe_lora_bwd(ctypes.byref(dd), ctypes.byref(rr), _ptr(dy), _ptr(W_gu), _ptr(A_gu), _ptr(B_gu),
                            _ptr(W_d), _ptr(A_d), _ptr(B_d), _ptr(saved), saved.numel(), _ptr(dx),
                            _ptr(dA_gu), _ptr(dB_gu), _ptr(dA_d), _ptr(dB_d), _ptr(d_topk_w), _ptr(workspace),
                            workspace.numel(), _ptr(dev_status), _stream(stream)))
    return dx, dA_gu, dB_gu, dA_d, dB_d


def moe_router_topk(logits: torch.Tensor, k: int, topk_idx=None, topk_w=None, stream=None):
    """Softmax over the E router logits of each token and its k largest
    probabilities (ties to the lower expert index); returns (topk_idx int32, topk_w)."""
    _need(logits, "logits", torch.float32)
    if logits.dim() != 2:
        raise MoEError("logits must be [T, E]")
    T, E = logits.shape
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _need(topk_idx, "topk_idx", torch.int32, (T, k))
    _need(topk_w, "topk_w", torch.float32, (T, k))
    _check(load_library().moe_router_topk(_ptr(logits), T, E, k, _ptr(topk_idx), _ptr(topk_w), _stream(stream)))
    return topk_idx, topk_w


@dataclass
class PackedMetadata:
    """Device-side metadata of one packed batch (moe_packed_metadata); nothing here is on the host."""
    cu_seqlens: torch.Tensor   # [T+1] int32: entries 0..n are the samples' first tokens, then T
    seq_id: torch.Tensor       # [T] int32: the sample of each token
    n_seqs: torch.Tensor       # [1] int32: the number of samples n
    max_seqlen: torch.Tensor   # [1] int32: the longest sample
    T: int


def moe_packed_metadata(position_ids: torch.Tensor, out: PackedMetadata | None = None, stream=None) -> PackedMetadata:
    """Samples of a packed batch from its position ids (a sample starts at token 0 and at
    every token whose position id is 0): cu_seqlens, seq_id, n and the longest sample, built
    on the device without a host synchronisation.  `out` (same T) reuses its buffers."""
    if not isinstance(position_ids, torch.Tensor) or position_ids.dtype not in (torch.int32, torch.int64):
        raise MoEError("position_ids must be an int32 or int64 torch.Tensor")
    pos = position_ids.reshape(-1)
    _need(pos, "position_ids", pos.dtype)
    T = pos.numel()
    dev = pos.device
    if out is not None:
        if out.T != T:
            raise MoEError(f"out holds metadata for {out.T} tokens, position_ids has {T}")
        cu, seq_id, n, mx = out.cu_seqlens, out.seq_id, out.n_seqs, out.max_seqlen
    else:
        cu = torch.empty(T + 1, dtype=torch.int32, device=dev)
        seq_id = torch.empty(T, dtype=torch.int32, device=dev)
        n = torch.empty(1, dtype=torch.int32, device=dev)
        mx = torch.empty(1, dtype=torch.int32, device=dev)
    _need(cu, "cu_seqlens", torch.int32, (T + 1,))
    _need(seq_id, "seq_id", torch.int32, (T,))
    _check(load_library().moe_packed_metadata(_ptr(pos), pos.element_size(), T, _ptr(cu), _ptr(seq_id), _ptr(n),
                                              _ptr(mx), _stream(stream)))
    return PackedMetadata(cu, seq_id, n, mx, T)


def moe_packed_causal_mask(meta: PackedMetadata, mask=None, stream=None) -> torch.Tensor:
    """The block-diagonal causal mask of a packed batch: mask[i, j] is True when tokens i
    and j lie in the same sample and j <= i (bool [T, T])."""
    T = meta.T
    if mask is None:
        mask = torch.empty((T, T), dtype=torch.bool, device=meta.seq_id.device)
    _need(mask, "mask", torch.bool, (T, T))
    _check(load_library().moe_packed_causal_mask(_ptr(meta.cu_seqlens), _ptr(meta.seq_id), T, _ptr(mask),
                                                 _stream(stream)))
    return mask


class PackedBatch:
    """Metadata of one packed batch, built once and reused by every layer.

    The device tensors are built on construction; the mask on its first request; the
    host integers (n, longest sample) on their first request, with the one host
    synchronisation that reading them costs, once per batch instead of once per layer.
    """

    def __init__(self, position_ids: torch.Tensor, stream=None):
        self.meta = moe_packed_metadata(position_ids, stream=stream)
        self._stream = stream
        self._mask = None
        self._host = None

    def causal_mask(self) -> torch.Tensor:
        if self._mask is None:
            self._mask = moe_packed_causal_mask(self.meta, stream=self._stream)
        return self._mask

    def host_sizes(self):
        """(n_seqs, max_seqlen) as Python ints, read from the device once."""
        if self._host is None:
            both = torch.cat([self.meta.n_seqs, self.meta.max_seqlen]).cpu()
            self._host = (int(both[0]), int(both[1]))
        return self._host

    def cu_seqlens(self) -> torch.Tensor:
        """cu_seqlens trimmed to its n + 1 valid entries (uses host_sizes)."""
        return self.meta.cu_seqlens[: self.host_sizes()[0] + 1]


def moe_router_bwd(logits: torch.Tensor, topk_idx: torch.Tensor, d_topk_w: torch.Tensor, d_logits=None,
                   stream=None) -> torch.Tensor:
    """Gradient of the router step w.r.t. the logits (selection held fixed)."""
    _need(logits, "logits", torch.float32)
    T, E = logits.shape
    k = topk_idx.shape[1]
    _need(topk_idx, "topk_idx", torch.int32, (T, k))
    _need(d_topk_w, "d_topk_w", torch.float32, (T, k))
    if d_logits is None:
        d_logits = torch.empty_like(logits)
    _need(d_logits, "d_logits", torch.float32, (T, E))
    _check(load_library().moe_router_bwd(_ptr(logits), _ptr(topk_idx), _ptr(d_topk_w), T, E, k, _ptr(d_logits),
                                         _stream(stream)))
    return d_logits


def moe_quantize_fp8(W: torch.Tensor, stream=None):
    """FP8 (e4m3) codes and per-column power-of-two scales of a bf16 weight stack
    [..., rows, cols]; returns (Wq uint8, scales float32 [..., cols])."""
    _need(W, "W", torch.bfloat16)
    rows, cols = W.shape[-2], W.shape[-1]
    n_mat = W.numel() // max(rows * cols, 1)
    Wq = torch.empty(W.shape, dtype=torch.uint8, device=W.device)
    sc = torch.empty(W.shape[:-2] + (cols,), dtype=torch.float32, device=W.device)
    _check(load_library().moe_quantize_fp8(_ptr(W), n_mat, rows, cols, _ptr(Wq), _ptr(sc), _stream(stream)))
    return Wq, sc


def moe_quantize_nf4(W: torch.Tensor, stream=None):
    """NF4 codes (two per byte) and per-64-element absmax scales of a bf16 weight stack
    [..., rows, cols], cols a multiple of 64; returns (Wq uint8 [..., rows, cols / 2],
    absmax float32 [..., cols / 64, rows], block-major)."""
    _need(W, "W", torch.bfloat16)
    rows, cols = W.shape[-2], W.shape[-1]
    if cols % 64:
        raise MoEError("NF4 quantisation needs rows of a multiple of 64 elements")
    n_mat = W.numel() // max(rows * cols, 1)
    Wq = torch.empty(W.shape[:-1] + (cols // 2,), dtype=torch.uint8, device=W.device)
    am = torch.empty(W.shape[:-2] + (cols // 64, rows), dtype=torch.float32, device=W.device)
    _check(load_library().moe_quantize_nf4(_ptr(W), n_mat, rows, cols, _ptr(Wq), _ptr(am), _stream(stream)))
    return Wq, am


def moe_nf4_codebook() -> list:
    """The 16 NF4 code values the library quantises and dequantises with (ascending)."""
    buf = (ctypes.c_float * 16)()
    _check(load_library().moe_nf4_codebook(buf))
    return list(buf)


def quantize_expert_weights(weights: dict, stream=None, fmt: str = "fp8") -> dict:
    """Expert weights with the two base stacks replaced by codes + scales: fmt "fp8" (e4m3
    codes, column scales: keys Wq_gu, s_gu, Wq_d, s_d) or "nf4" (4-bit NormalFloat codes,
    64-element block scales: keys W4_gu, m_gu, W4_d, m_d)."""
    out = {k: v for k, v in weights.items() if k not in ("W_gu", "W_d")}
    if fmt == "fp8":
        out["Wq_gu"], out["s_gu"] = moe_quantize_fp8(weights["W_gu"], stream)
        out["Wq_d"], out["s_d"] = moe_quantize_fp8(weights["W_d"], stream)
    elif fmt == "nf4":
        out["W4_gu"], out["m_gu"] = moe_quantize_nf4(weights["W_gu"], stream)
        out["W4_d"], out["m_d"] = moe_quantize_nf4(weights["W_d"], stream)
    else:
        raise MoEError(f"unknown weight format {fmt!r}")
    return out


def _lora_factor_checks(d: Dims, w: dict):
    bf = torch.bfloat16
    _need(w["A_gu"], "A_gu", bf, (d.E, d.r, d.H))
    _need(w["B_gu"], "B_gu", bf, (d.E, d.r, 2 * d.I))
    _need(w["A_d"], "A_d", bf, (d.E, d.r, d.I))
    _need(w["B_d"], "B_d", bf, (d.E, d.r, d.H))


def _fp8_args(d: Dims, w: dict):
    _need(w["Wq_gu"], "Wq_gu", torch.uint8, (d.E, d.H, 2 * d.I))
    _need(w["s_gu"], "s_gu", torch.float32, (d.E, 2 * d.I))
    _need(w["Wq_d"], "Wq_d", torch.uint8, (d.E, d.I, d.H))
    _need(w["s_d"], "s_d", torch.float32, (d.E, d.H))
    _lora_factor_checks(d, w)
    return [_ptr(w[n]) for n in ("Wq_gu", "s_gu", "A_gu", "B_gu", "Wq_d", "s_d", "A_d", "B_d")]


def _nf4_args(d: Dims, w: dict):
    _need(w["W4_gu"], "W4_gu", torch.uint8, (d.E, d.H, d.I))
    _need(w["m_gu"], "m_gu", torch.float32, (d.E, 2 * d.I // 64, d.H))
    _need(w["W4_d"], "W4_d", torch.uint8, (d.E, d.I, d.H // 2))
    _need(w["m_d"], "m_d", torch.float32, (d.E, d.H // 64, d.I))
    _lora_factor_checks(d, w)
    return [_ptr(w[n]) for n in ("W4_gu", "m_gu", "A_gu", "B_gu", "W4_d", "m_d", "A_d", "B_d")]


def moe_lora_fwd_fp8(d: Dims, rt: Routing, x, w: dict, y, saved, workspace, dev_status, stream=None):
    """Forward with FP8 base weights (`w` from quantize_expert_weights)."""
    _need(x, "x", torch.bfloat16, (d.T, d.H))
    dd, rr = d.c_struct(), rt.c_struct()
    _check(load_library().moe_lora_fwd_fp8(ctypes.byref(dd), ctypes.byref(rr), _ptr(x), *_fp8_args(d, w), _ptr(y),
                                           _ptr(saved), saved.numel(), _ptr(workspace), workspace.numel(),
                                           _ptr(dev_status), _stream(stream)))
    return y


def moe_lora_bwd_fp8(d: Dims, rt: Routing, dy, w: dict, saved, dx, grads, workspace, dev_status, stream=None,
                     d_topk_w=None):
    """Backward with FP8 base weights; returns (dx, dA_gu, dB_gu, dA_d, dB_d)."""
    _need(dy, "dy", torch.bfloat16, (d.T, d.H))
    dA_gu, dB_gu, dA_d, dB_d = grads
    dd, rr = d.c_struct(), rt.c_struct()
    _check(load_library().moe_lora_bwd_fp8(ctypes.byref(dd), ctypes.byref(rr), _ptr(dy), *_fp8_args(d, w),
                                           _ptr(saved), saved.numel(), _ptr(dx), _ptr(dA_gu), _ptr(dB_gu),
                                           _ptr(dA_d), _ptr(dB_d), _ptr(d_topk_w), _ptr(workspace),
                                           workspace.numel(), _ptr(dev_status), _stream(stream)))
    return dx, dA_gu, dB_gu, dA_d, dB_d


def moe_lora_fwd_nf4(d: Dims, rt: Routing, x, w: dict, y, saved, workspace, dev_status, stream=None):
    """Forward with NF4 base weights (`w` from quantize_expert_weights(..., fmt="nf4"))."""
    _need(x, "x", torch.bfloat16, (d.T, d.H))
    dd, rr = d.c_struct(), rt.c_struct()
    _check(load_library().moe_lora_fwd_nf4(ctypes.byref(dd), ctypes.byref(rr), _ptr(x), *_nf4_args(d, w), _ptr(y),
                                           _ptr(saved), saved.numel(), _ptr(workspace), workspace.numel(),
                                           _ptr(dev_status), _stream(stream)))
    return y


def moe_lora_bwd_nf4(d: Dims, rt: Routing, dy, w: dict, saved, dx, grads, workspace, dev_status, stream=None,
                     d_topk_w=None):
    """Backward with NF4 base weights; returns (dx, dA_gu, dB_gu, dA_d, dB_d)."""
    _need(dy, "dy", torch.bfloat16, (d.T, d.H))
    dA_gu, dB_gu, dA_d, dB_d = grads
    dd, rr = d.c_struct(), rt.c_struct()
    _check(load_library().moe_lora_bwd_nf4(ctypes.byref(dd), ctypes.byref(rr), _ptr(dy), *_nf4_args(d, w),
                                           _ptr(saved), saved.numel(), _ptr(dx), _ptr(dA_gu), _ptr(dB_gu),
                                           _ptr(dA_d), _ptr(dB_d), _ptr(d_topk_w), _ptr(workspace),
                                           workspace.numel(), _ptr(dev_status), _stream(stream)))
    return dx, dA_gu, dB_gu, dA_d, dB_d


def moe_launch_count() -> int:
    """Launch operations the library has issued so far (host-side count)."""
    return int(load_library().moe_launch_count())


def moe_diag_force_timeout(launch_index: int, limit_ns: int = 1_000_000) -> None:
    """Make the launch_index-th single-CTA tensor-core launch from now give up its waits
    (failure-path test hook of the C ABI; launch_index < 0 disarms)."""
    _check(load_library().moe_diag_force_timeout(int(launch_index), int(limit_ns)))


def moe_timing_enable(on: bool) -> None:
    """Start (clearing the record) or stop per-kernel event timing."""
    _check(load_library().moe_timing_enable(1 if on else 0))


def moe_timing_read() -> dict:
    """{kernel name: (total ms, launches)} of the launches recorded since the last
    moe_timing_enable(True).  Waits for the recorded events."""
    lib = load_library()
    out = {}
    buf = ctypes.create_string_buffer(64)
    ms, n = ctypes.c_double(), ctypes.c_int32()
    i = 0
    while True:
        st = lib.moe_timing_read(i, buf, 64, ctypes.byref(ms), ctypes.byref(n))
        if st == 2:
            break
        _check(st)
        out[buf.value.decode()] = (ms.value, n.value)
        i += 1
    return out


class MoELoRALayer:
    """Preallocated buffers for repeated route + forward + backward calls on one
    stream (no allocation inside a step, so a step can be graph-captured).
    `weights`: the bf16 expert weights, or those of quantize_expert_weights (FP8 or NF4
    base; the layer then calls the _fp8 / _nf4 entry points).
    h_from_gu: bf16 weights only; the forward forms h from the stored bf16 GU
    (moe_lora_fwd_h_from_gu), as the offloaded stack does."""

    def __init__(self, d: Dims, weights: dict, device="cuda", h_from_gu=False):
        self.d = d
        self.w = weights
        self.h_from_gu = h_from_gu
        self.fp8 = "Wq_gu" in weights          # FP8 base weights (quantize_expert_weights)
        self.nf4 = "W4_gu" in weights          # NF4 base weights (quantize_expert_weights, fmt="nf4")
        if h_from_gu and (self.fp8 or self.nf4):
            raise MoEError("h_from_gu is a forward of the bf16 weights only")
        dev = torch.device(device)
        self.rt = Routing.empty(d.T, d.k, d.E, dev)
        self.route_ws = torch.empty(moe_route_workspace_size(d.T, d.k, d.E), dtype=torch.uint8, device=dev)
        sb, wb = moe_lora_fwd_sizes(d)
        self.saved = torch.empty(max(sb, 16), dtype=torch.uint8, device=dev)
        self.fwd_ws = torch.empty(max(wb, 16), dtype=torch.uint8, device=dev)
        self.bwd_ws = torch.empty(max(moe_lora_bwd_workspace_size(d), 16), dtype=torch.uint8, device=dev)
        self.y = torch.empty((d.T, d.H), dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty((d.T, d.H), dtype=torch.bfloat16, device=dev)
        self.grads = tuple(torch.empty_like(weights[n]) for n in ("A_gu", "B_gu", "A_d", "B_d"))
        self.d_topk_w = torch.empty((d.T, d.k), dtype=torch.float32, device=dev)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)

    def _wts(self):
        w = self.w
        return w["W_gu"], w["A_gu"], w["B_gu"], w["W_d"], w["A_d"], w["B_d"]

    def route(self, topk_idx, topk_w, stream=None):
        return moe_route(topk_idx, topk_w, self.d.E, out=self.rt, workspace=self.route_ws,
                         dev_status=self.dev_status, stream=stream)

    def forward(self, x, stream=None):
        if self.fp8:
            return moe_lora_fwd_fp8(self.d, self.rt, x, self.w, self.y, self.saved, self.fwd_ws, self.dev_status,
                                    stream)
        if self.nf4:
            return moe_lora_fwd_nf4(self.d, self.rt, x, self.w, self.y, self.saved, self.fwd_ws, self.dev_status,
                                    stream)
        return moe_lora_fwd(self.d, self.rt, x, *self._wts(), y=self.y, saved=self.saved,
                            workspace=self.fwd_ws, dev_status=self.dev_status, stream=stream,
                            h_from_gu=self.h_from_gu)[0]

    def backward(self, dy, stream=None, with_topk_grad=True):
        dtw = self.d_topk_w if with_topk_grad else None
        if self.fp8:
            return moe_lora_bwd_fp8(self.d, self.rt, dy, self.w, self.saved, self.dx, self.grads, self.bwd_ws,
                                    self.dev_status, stream, d_topk_w=dtw)
        if self.nf4:
            return moe_lora_bwd_nf4(self.d, self.rt, dy, self.w, self.saved, self.dx, self.grads, self.bwd_ws,
                                    self.dev_status, stream, d_topk_w=dtw)
        return moe_lora_bwd(self.d, self.rt, dy, *self._wts(), self.saved, dx=self.dx, grads=self.grads,
                            workspace=self.bwd_ws, dev_status=self.dev_status, stream=stream, d_topk_w=dtw)

    def step(self, topk_idx, topk_w, x, dy, stream=None, with_topk_grad=True):
        self.route(topk_idx, topk_w, stream)
        self.forward(x, stream)
        return self.backward(dy, stream, with_topk_grad)
