"""GB300-native (sm_103a) MoE-LoRA expert layer.

Routing (histogram, scan, stable scatter), Split-LoRA grouped GEMMs with a
fused SwiGLU, a deterministic routing-weighted combine and the backward for
dx and the per-expert LoRA gradients, all in hand-written CUDA behind the C
ABI declared in ``include/moe_lora.h``.  ``binding`` is the Python side of
that ABI; importing this package does not load the library.
"""
from .binding import (  # noqa: F401
    Dims, MoEError, MoELoRALayer, Routing, load_library, moe_lora_bwd, moe_lora_bwd_fp8, moe_lora_bwd_workspace_size,
    moe_lora_fwd_fp8, moe_quantize_fp8, quantize_expert_weights,
    moe_lora_fwd_nf4, moe_lora_bwd_nf4, moe_quantize_nf4, moe_nf4_codebook,
    moe_launch_count, moe_lora_fwd, moe_lora_fwd_sizes, moe_lora_saved_layout, moe_lora_saved_regather, moe_lora_saved_rebuild_h, moe_route, moe_route_workspace_size, moe_router_bwd, moe_router_topk, moe_timing_enable,
    moe_timing_read, moe_diag_force_timeout, PackedBatch, PackedMetadata, moe_packed_metadata, moe_packed_causal_mask,
)
