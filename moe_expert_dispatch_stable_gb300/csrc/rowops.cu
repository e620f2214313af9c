// Row kernels of the MoE-LoRA layer: the permuted-row gather (with the
// routing-weight scale for the backward) and the deterministic per-token
// combine.  Both are HBM-bound copies with at most one flop per element.
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace moe {

namespace {

int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!cached[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = v > 0 ? v : 1;
    }
    return cached[dev];
}

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 pack8(const float* f) {
    uint4 v;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return v;
}

}  // namespace

// ---------------------------------------------------------------- gather
// One warp per sorted row: dst[p] = src[perm[p] / k] (x k-fold, in expert order).
__global__ void gather_rows_kernel(const uint4* __restrict__ src, int vpr, const int32_t* __restrict__ perm,
                                   const float* __restrict__ w_sorted, int64_t N, int k,
                                   uint4* __restrict__ dst) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t p = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < N; p += nwarps) {
        const int64_t t = perm[p] / k;
        const uint4* s = src + t * vpr;
        uint4* d = dst + p * vpr;
        if (w_sorted == nullptr) {
            for (int v = lane; v < vpr; v += 32) d[v] = __ldg(s + v);
        } else {
            const float w = w_sorted[p];
            for (int v = lane; v < vpr; v += 32) {
                float f[8];
                unpack8(__ldg(s + v), f);
#pragma unroll
                for (int i = 0; i < 8; ++i) f[i] *= w;
                d[v] = pack8(f);
            }
        }
    }
}

cudaError_t launch_gather_rows(const void* src, int H, const int32_t* perm, const float* w_sorted,
                               int64_t N, int k, void* dst, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>((N + 7) / 8, (int64_t)num_sms() * 16);
    gather_rows_kernel<<<(unsigned)blocks, threads, 0, s>>>((const uint4*)src, H / 8, perm, w_sorted, N, k,
                                                           (uint4*)dst);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- combine
// One warp per token: out[t] = sum_{j=0}^{k-1} src[inv_perm[t*k+j]] in that order.
__global__ void combine_kernel(const float4* __restrict__ src, const int32_t* __restrict__ inv_perm,
                               int64_t T, int k, int vpr4, uint2* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
        for (int v = lane; v < vpr4; v += 32) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j = 0; j < k; ++j) {
                const int64_t row = inv_perm[t * k + j];
                const float4 a = __ldg(src + row * vpr4 + v);
                acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
            }
            uint2 o;
            __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
            h[0] = __floats2bfloat162_rn(acc.x, acc.y);
            h[1] = __floats2bfloat162_rn(acc.z, acc.w);
            out[t * vpr4 + v] = o;
        }
    }
}

cudaError_t launch_combine(const float* src, const int32_t* inv_perm, int64_t T, int k, int H,
                           void* out, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>((T + 7) / 8, (int64_t)num_sms() * 16);
    combine_kernel<<<(unsigned)blocks, threads, 0, s>>>((const float4*)src, inv_perm, T, k, H / 4, (uint2*)out);
    return cudaGetLastError();
}

}  // namespace moe
