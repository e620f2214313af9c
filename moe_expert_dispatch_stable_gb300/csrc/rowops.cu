// Row kernels of the MoE-LoRA layer: the permuted-row gather (with the
// routing-weight scale and the routing-weight gradient for the backward) and
// the deterministic, routing-weighted per-token combine.  Both are HBM-bound,
// with a couple of flops per element.
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
// One warp per sorted row: dst[p] = src[perm[p] / k] (x k-fold, in expert order),
// optionally scaled by the row's routing weight.  With O / d_w: the backward's
// routing-weight gradient d_w[perm[p]] = <src row, O[p]> (the unweighted expert
// output of the slot), accumulated in fp32 while the row is in registers.
__global__ void gather_rows_kernel(const uint4* __restrict__ src, int vpr, const int32_t* __restrict__ perm,
                                   const float* __restrict__ w_sorted, int64_t N, int k,
                                   uint4* __restrict__ dst, const uint4* __restrict__ O, float* __restrict__ d_w) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t p = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < N; p += nwarps) {
        const int slot = perm[p];
        const int64_t t = slot / k;
        const uint4* s = src + t * vpr;
        uint4* d = dst + p * vpr;
        if (w_sorted == nullptr) {
            for (int v = lane; v < vpr; v += 32) d[v] = __ldg(s + v);
        } else {
            const float w = w_sorted[p];
            float dot = 0.f;
            for (int v = lane; v < vpr; v += 32) {
                float f[8];
                unpack8(__ldg(s + v), f);
                if (d_w != nullptr) {
                    float o[8];
                    unpack8(__ldcs(O + p * vpr + v), o);
#pragma unroll
                    for (int i = 0; i < 8; ++i) dot = fmaf(f[i], o[i], dot);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) f[i] *= w;
                d[v] = pack8(f);
            }
            if (d_w != nullptr) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
                if (lane == 0) d_w[slot] = dot;
            }
        }
    }
}

cudaError_t launch_gather_rows(const void* src, int H, const int32_t* perm, const float* w_sorted,
                               int64_t N, int k, void* dst, const void* O, float* d_w, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>((N + 7) / 8, (int64_t)num_sms() * 16);
    gather_rows_kernel<<<(unsigned)blocks, threads, 0, s>>>((const uint4*)src, H / 8, perm, w_sorted, N, k,
                                                           (uint4*)dst, (const uint4*)O, d_w);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- combine
// One warp per token: out[t] = sum_{j=0}^{k-1} src[inv_perm[t*k+j]] in that order,
// summed in fp32, 8 columns per lane per step (bf16 or fp32 source rows).
template <typename SrcT>
__device__ __forceinline__ void load8(const SrcT* row, int v, float* a);

template <>
__device__ __forceinline__ void load8<bf16>(const bf16* row, int v, float* a) {
    unpack8(__ldcs(reinterpret_cast<const uint4*>(row) + v), a);
}

template <>
__device__ __forceinline__ void load8<float>(const float* row, int v, float* a) {
    const float4 lo = __ldcs(reinterpret_cast<const float4*>(row) + 2 * v);
    const float4 hi = __ldcs(reinterpret_cast<const float4*>(row) + 2 * v + 1);
    a[0] = lo.x; a[1] = lo.y; a[2] = lo.z; a[3] = lo.w;
    a[4] = hi.x; a[5] = hi.y; a[6] = hi.z; a[7] = hi.w;
}

template <typename SrcT>
__global__ void combine_kernel(const SrcT* __restrict__ src, const float* __restrict__ w_sorted,
                               const int32_t* __restrict__ inv_perm, int64_t T, int k, int H,
                               uint4* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int vpr = H / 8;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
        for (int v = lane; v < vpr; v += 32) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int j = 0; j < k; ++j) {
                const int64_t row = inv_perm[t * k + j];
                const float w = w_sorted != nullptr ? w_sorted[row] : 1.0f;
                float a[8];
                load8<SrcT>(src + row * H, v, a);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(w, a[i], acc[i]);
            }
            out[t * vpr + v] = pack8(acc);
        }
    }
}

cudaError_t launch_combine(const void* src, bool src_f32, const float* w_sorted, const int32_t* inv_perm, int64_t T,
                           int k, int H, void* out, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>((T + 7) / 8, (int64_t)num_sms() * 16);
    if (src_f32)
        combine_kernel<float><<<(unsigned)blocks, threads, 0, s>>>((const float*)src, w_sorted, inv_perm, T, k, H,
                                                                   (uint4*)out);
    else
        combine_kernel<bf16><<<(unsigned)blocks, threads, 0, s>>>((const bf16*)src, w_sorted, inv_perm, T, k, H,
                                                                  (uint4*)out);
    return cudaGetLastError();
}

}  // namespace moe
