"""Offloaded activations for a stack of MoE-LoRA layers, reloaded double-buffered.

The Unsloth x NVIDIA blog post (section "core idea / structure / how it
works", double-buffered checkpoint reload) keeps activations in pinned host
memory and brings them back for the backward pass on a copy stream: while the
backward computes with buffer A, the next layer's activations are copied into
buffer B, and the two swap roles; the extra buffer is only used when the VRAM
budget allows, otherwise a single buffer (copy, wait, compute) is used.

Applied here to the `saved` buffer of each MoE-LoRA layer of a stack
x_{l+1} = MoE_l(x_l): after layer l's forward its saved activations are copied
to pinned host memory (the device buffer is then reused by the next layer), and
the backward walks the layers in reverse, reloading layer l-1's activations
while layer l's backward runs.  Only stream-ordered copies and events are used:
no host synchronisation inside forward() or backward().

Only the sections the backward cannot rebuild exactly cross the host link: GU, XA_s
and HA_s.  x_perm is regathered on the device from the layer's input
(moe_lora_saved_regather, bit-identical to the forward's gather), h is rebuilt from GU
(moe_lora_saved_rebuild_h: the stack's forward, moe_lora_fwd_h_from_gu, forms h from the
stored bf16 GU with the same arithmetic, so the rebuild is bit-identical), and O, which
only the router's d topk_w
reads, is not needed because the stack returns no router gradients.  That is 60 % fewer
bytes than the whole saved buffer for the GPT-OSS-20B-shaped layer, whose reload is
bound by the ~200 GB/s host-to-device link.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import binding as B


@dataclass(frozen=True)
class ReloadStep:
    layer: int      # layer whose saved activations are reloaded
    buffer: int     # device buffer they are reloaded into
    after: int      # layer whose backward must have finished with that buffer (-1: none)


def reload_schedule(n_layers: int, n_buffers: int) -> list[ReloadStep]:
    """Order of the reloads of the backward pass (layers L-1 .. 0).

    Layer l uses buffer (L-1-l) % n_buffers.  A reload may start once the layer that
    last used its buffer has finished its backward; with two buffers that is the layer
    two steps later in the backward, so reload l-1 overlaps the backward of l."""
    if n_layers < 1 or n_buffers < 1:
        raise ValueError("need at least one layer and one buffer")
    out = []
    for i, l in enumerate(range(n_layers - 1, -1, -1)):
        prev = i - n_buffers
        out.append(ReloadStep(layer=l, buffer=i % n_buffers,
                              after=(n_layers - 1 - prev) if prev >= 0 else -1))
    return out


def choose_buffers(saved_bytes: int, free_bytes: int, reserve_bytes: int, want: int = 2) -> int:
    """VRAM guardrail: use the second buffer only if it fits with `reserve_bytes` to spare."""
    if want >= 2 and free_bytes - 2 * saved_bytes >= reserve_bytes:
        return 2
    if free_bytes - saved_bytes >= 0:
        return 1
    raise MemoryError("not enough device memory for one saved-activation buffer")


class OffloadedMoEStack:
    """L MoE-LoRA layers with host-offloaded saved activations.

    weights: list of L dicts (W_gu, A_gu, B_gu, W_d, A_d, B_d on the device).
    buffers: 2 (double-buffered reload), 1 (copy, then compute), or "auto" (two if
    they fit the VRAM budget: free memory minus `reserve_bytes`).
    The input of forward() must stay unchanged until backward() has run (x_perm of
    the first layer is regathered from it); the later layers' inputs are the stack's
    own outputs."""

    def __init__(self, d: B.Dims, weights: list, device="cuda", buffers="auto", reserve_bytes: int = 1 << 30):
        self.d = d
        self.w = weights
        self.L = len(weights)
        dev = torch.device(device)
        self.dev = dev
        saved_b, ws_b = B.moe_lora_fwd_sizes(d)
        self.saved_bytes = max(saved_b, 16)
        offs, _ = B.moe_lora_saved_layout(d)
        # the byte ranges [lo, hi) of `saved` that cross the host link: GU, then XA_s and
        # HA_s (h, between them, is rebuilt on the device); packed back to back on the host
        self.spans = [(offs[1], offs[2]), (offs[3], offs[5])]
        self.transfer_bytes = sum(hi - lo for lo, hi in self.spans)
        if buffers == "auto":
            free, _ = torch.cuda.mem_get_info(dev)
            self.n_buf = choose_buffers(self.saved_bytes, free, reserve_bytes)
        else:
            self.n_buf = int(buffers)
        self.bufs = [torch.empty(self.saved_bytes, dtype=torch.uint8, device=dev) for _ in range(self.n_buf)]
        self.host = [torch.empty(max(self.transfer_bytes, 16), dtype=torch.uint8).pin_memory() for _ in range(self.L)]
        self._x_in = [None] * self.L
        self.fwd_ws = torch.empty(max(ws_b, 16), dtype=torch.uint8, device=dev)
        self.bwd_ws = torch.empty(max(B.moe_lora_bwd_workspace_size(d), 16), dtype=torch.uint8, device=dev)
        self.route_ws = torch.empty(B.moe_route_workspace_size(d.T, d.k, d.E), dtype=torch.uint8, device=dev)
        self.rt = [B.Routing.empty(d.T, d.k, d.E, dev) for _ in range(self.L)]
        self.y = [torch.empty((d.T, d.H), dtype=torch.bfloat16, device=dev) for _ in range(self.L)]
        self.dx = [torch.empty((d.T, d.H), dtype=torch.bfloat16, device=dev) for _ in range(self.L)]
        self.grads = [tuple(torch.empty_like(wl[n]) for n in ("A_gu", "B_gu", "A_d", "B_d")) for wl in weights]
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.copy_stream = torch.cuda.Stream(dev)
        self._copied = [torch.cuda.Event() for _ in range(self.L)]       # D2H of layer l done
        self._reloaded = [torch.cuda.Event() for _ in range(self.L)]     # H2D of layer l done
        self._bwd_done = [torch.cuda.Event() for _ in range(self.L)]     # backward of layer l done

    def _wts(self, l):
        w = self.w[l]
        return w["W_gu"], w["A_gu"], w["B_gu"], w["W_d"], w["A_d"], w["B_d"]

    def forward(self, x, routing):
        """routing: list of (topk_idx, topk_w) per layer.  Returns the last layer's y."""
        comp = torch.cuda.current_stream(self.dev)
        for l in range(self.L):
            buf = self.bufs[l % self.n_buf]
            if l >= self.n_buf:
                comp.wait_event(self._copied[l - self.n_buf])   # the D2H of this buffer's last user is done
            B.moe_route(routing[l][0], routing[l][1], self.d.E, out=self.rt[l], workspace=self.route_ws,
                        dev_status=self.dev_status)
            B.moe_lora_fwd(self.d, self.rt[l], x, *self._wts(l), y=self.y[l], saved=buf,
                           workspace=self.fwd_ws, dev_status=self.dev_status, h_from_gu=True)
            self._x_in[l] = x
            self.copy_stream.wait_stream(comp)
            with torch.cuda.stream(self.copy_stream):
                at = 0
                for lo, hi in self.spans:
                    self.host[l][at:at + hi - lo].copy_(buf[lo:hi], non_blocking=True)
                    at += hi - lo
                self._copied[l].record(self.copy_stream)
            x = self.y[l]
        return x

    def backward(self, dy):
        """Reverse pass with the saved activations reloaded from host memory."""
        comp = torch.cuda.current_stream(self.dev)
        plan = reload_schedule(self.L, self.n_buf)
        by_layer = {s.layer: s for s in plan}

        def issue_reload(step: ReloadStep):
            with torch.cuda.stream(self.copy_stream):
                self.copy_stream.wait_event(self._copied[step.layer])
                if step.after >= 0:
                    self.copy_stream.wait_event(self._bwd_done[step.after])
                at = 0
                for lo, hi in self.spans:
                    self.bufs[step.buffer][lo:hi].copy_(self.host[step.layer][at:at + hi - lo], non_blocking=True)
                    at += hi - lo
                self._reloaded[step.layer].record(self.copy_stream)

        # prime the pipeline: as many reloads as there are buffers
        for step in plan[: self.n_buf]:
            issue_reload(step)
        issued = min(self.n_buf, self.L)
        for i, l in enumerate(range(self.L - 1, -1, -1)):
            step = by_layer[l]
            comp.wait_event(self._reloaded[l])
            B.moe_lora_saved_regather(self.d, self.rt[l], self._x_in[l], self.bufs[step.buffer])
            B.moe_lora_saved_rebuild_h(self.d, self.bufs[step.buffer])
            B.moe_lora_bwd(self.d, self.rt[l], dy, *self._wts(l), self.bufs[step.buffer], dx=self.dx[l],
                           grads=self.grads[l], workspace=self.bwd_ws, dev_status=self.dev_status)
            self._bwd_done[l].record(comp)
            if issued < self.L:
                issue_reload(plan[issued])
                issued += 1
            dy = self.dx[l]
        return dy
