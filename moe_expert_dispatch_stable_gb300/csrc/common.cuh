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

// ---- programmatic dependent launch
// The library's kernels are launched with programmatic stream serialisation, so that a
// kernel's launch overlaps the tail of the kernel before it on the stream.  Every kernel
// starts with pdl_wait() (before any global-memory access or TMEM allocation: it then sees
// every result of the previous kernel, exactly as with plain stream order).  The short
// kernels (routing, gathers, combines, router) then call pdl_trigger(), so the next
// kernel's launch proceeds while they run; the grouped GEMMs do not, since CTAs of the
// next kernel waiting through a GEMM's whole duration measured slower.  Both are no-ops
// for a kernel launched without the attribute.  Measured: the T = 64 layer's step
// 0.114 -> 0.077 ms, the Qwen3-30B-shaped step 1.71 -> 1.67 ms.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// ---- debug build
// With MOE_DEBUG=1 (a separate build of the library) every index read from a caller's
// routing buffer is checked before it is used: an index outside [0, n) sets
// MOE_DEV_BAD_INDEX in the status word (when the call has one) and the access is skipped.
// No trap, no assert.  The release build (MOE_DEBUG=0) compiles the checks away.
#ifndef MOE_DEBUG
#define MOE_DEBUG 0
#endif

__device__ __forceinline__ bool dbg_index_ok(int64_t i, int64_t n, int32_t* status) {
    if (!MOE_DEBUG || (i >= 0 && i < n)) return true;
    if (status != nullptr) atomicOr(status, MOE_DEV_BAD_INDEX);
    return false;
}

// Debug build: offsets [E+1] must start at 0, never decrease and end at N; tile offsets
// (when given) must count ceil(rows / tile_m) tiles per expert.  Checked by one thread.
__device__ __forceinline__ bool dbg_offsets_ok(const int32_t* offs, const int32_t* toffs, int E, int64_t N, int tile_m,
                                               int32_t* status) {
    if (!MOE_DEBUG) return true;
    bool ok = offs[0] == 0 && offs[E] == N && (toffs == nullptr || toffs[0] == 0);
    for (int e = 0; e < E && ok; ++e) {
        ok = offs[e + 1] >= offs[e];
        if (ok && toffs != nullptr) ok = toffs[e + 1] - toffs[e] == (offs[e + 1] - offs[e] + tile_m - 1) / tile_m;
    }
    if (!ok && status != nullptr) atomicOr(status, MOE_DEV_BAD_INDEX);
    return ok;
}

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
