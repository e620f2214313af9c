// Router in front of the routing: softmax over the E logits of a token, the k
// largest probabilities (descending, ties to the lower expert index, no
// renormalisation), and the backward of that step (the softmax VJP with the
// selection held fixed).
//
// The MoE-LoRA workloads route each token by "softmax, then top-k" over its
// router logits.  Softmax is strictly increasing in each logit, so the
// selection is made on the fp32 logits themselves (exact comparisons), and
// only the selected probabilities are computed: p_e = exp(z_e - max) / sum.
//
// One warp per token; the token's logits are staged in shared memory and the k
// winners are found by k warp-wide arg-max rounds over a selected-bit mask.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>
#include <mutex>

namespace moe {

namespace {

constexpr int kRouterWarps = 8;

// (value, index) order of the top-k: larger value first, then lower index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, d);
        const int oi = __shfl_xor_sync(0xffffffffu, i, d);
        if (better(ov, oi, v, i)) {
            v = ov;
            i = oi;
        }
    }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
    return v;
}

}  // namespace

__global__ void __launch_bounds__(32 * kRouterWarps)
router_topk_kernel(const float* __restrict__ logits, int64_t T, int E, int k, int32_t* __restrict__ topk_idx,
                   float* __restrict__ topk_w) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ float zsh[];                              // [kRouterWarps][E] + masks
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* z = zsh + warp * E;
    uint32_t* sel = reinterpret_cast<uint32_t*>(zsh + kRouterWarps * E) + warp * 32;
    for (int64_t t = (int64_t)blockIdx.x * kRouterWarps + warp; t < T; t += (int64_t)gridDim.x * kRouterWarps) {
        const float* row = logits + t * E;
        float m = -INFINITY;
        for (int e = lane; e < E; e += 32) {
            const float v = row[e];
            z[e] = v;
            m = fmaxf(m, v);
        }
        sel[lane] = 0u;
        m = warp_max(m);
        float s = 0.f;
        for (int e = lane; e < E; e += 32) s += expf(z[e] - m);
        s = warp_sum(s);
        __syncwarp();
        for (int j = 0; j < k; ++j) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            for (int e = lane; e < E; e += 32) {
                if (sel[e >> 5] & (1u << (e & 31))) continue;
                if (better(z[e], e, bv, bi)) {
                    bv = z[e];
                    bi = e;
                }
            }
            warp_argmax(bv, bi);
            if (lane == 0) {
                topk_idx[t * k + j] = bi;
                topk_w[t * k + j] = expf(bv - m) / s;
                sel[bi >> 5] |= 1u << (bi & 31);
            }
            __syncwarp();
        }
    }
}

// dz[t, e] = p_e * (g_e - sum_j dw[t,j] * p_{idx[t,j]}),  g_e = dw[t,j] where idx[t,j] = e.
__global__ void __launch_bounds__(32 * kRouterWarps)
router_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ topk_idx,
                  const float* __restrict__ d_topk_w, int64_t T, int E, int k, float* __restrict__ d_logits) {
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int64_t t = (int64_t)blockIdx.x * kRouterWarps + warp; t < T; t += (int64_t)gridDim.x * kRouterWarps) {
        const float* row = logits + t * E;
        float m = -INFINITY;
        for (int e = lane; e < E; e += 32) m = fmaxf(m, row[e]);
        m = warp_max(m);
        float s = 0.f;
        for (int e = lane; e < E; e += 32) s += expf(row[e] - m);
        s = warp_sum(s);
        const float inv = 1.0f / s;
        // c = sum_j dw_j * p_{idx_j}
        float c = 0.f;
        for (int j = lane; j < k; j += 32) {
            const int ix = topk_idx[t * k + j];
            if (dbg_index_ok(ix, E, nullptr)) c += d_topk_w[t * k + j] * expf(row[ix] - m) * inv;
        }
        c = warp_sum(c);
        for (int e = lane; e < E; e += 32) {
            float g = 0.f;
            for (int j = 0; j < k; ++j)
                if (topk_idx[t * k + j] == e) g = d_topk_w[t * k + j];
            const float p = expf(row[e] - m) * inv;
            d_logits[t * E + e] = p * (g - c);
        }
    }
}

cudaError_t launch_router_topk(const float* logits, int64_t T, int E, int k, int32_t* topk_idx, float* topk_w,
                               cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const size_t smem = (size_t)kRouterWarps * E * sizeof(float) + kRouterWarps * 32 * sizeof(uint32_t);
    // raise the kernel's dynamic shared-memory limit only when a call needs more than before
    {
        static std::mutex mu;
        static int granted[64] = {0};
        int dev = 0;
        cudaGetDevice(&dev);
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64 || (int)smem > granted[dev]) {
            cudaError_t e =
                cudaFuncSetAttribute(router_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) granted[dev] = (int)smem;
        }
    }
    const int64_t blocks = std::min<int64_t>((T + kRouterWarps - 1) / kRouterWarps, 152 * 16);
    return launch_pdl(router_topk_kernel, dim3((unsigned)blocks), dim3(32 * kRouterWarps), smem, s, logits, T, E, k,
                      topk_idx, topk_w);
}

cudaError_t launch_router_bwd(const float* logits, const int32_t* topk_idx, const float* d_topk_w, int64_t T, int E,
                              int k, float* d_logits, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((T + kRouterWarps - 1) / kRouterWarps, 152 * 16);
    return launch_pdl(router_bwd_kernel, dim3((unsigned)blocks), dim3(32 * kRouterWarps), 0, s, logits, topk_idx,
                      d_topk_w, T, E, k, d_logits);
}

}  // namespace moe
