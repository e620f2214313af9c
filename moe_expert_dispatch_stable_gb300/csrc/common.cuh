// Shared device helpers of the MoE-LoRA CUDA library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe_lora.h"

namespace moe {

using bf16 = __nv_bfloat16;

constexpr int kTileM = MOE_TILE_M;

__device__ __forceinline__ float bf2f(bf16 v) { return __bfloat162float(v); }
__device__ __forceinline__ bf16 f2bf(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

// Rounded-up padded LoRA rank used for the [N, RP] rank-r activations.
inline int lora_rp(int r) { return r <= 16 ? 16 : (r <= 32 ? 32 : 64); }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Expert owning sorted row p: largest e with offsets[e] <= p (offsets in smem).
__device__ __forceinline__ int expert_of_row(const int32_t* offs, int E, int p) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (offs[mid] <= p) lo = mid; else hi = mid - 1;
    }
    return lo;
}

}  // namespace moe
