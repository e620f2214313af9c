// Row kernels of the MoE-LoRA layer: permuted-row gather, deterministic
// per-token combine, rank-r LoRA projections and per-expert LoRA weight
// gradients.  All of them are HBM-bound (a handful of flops per byte).
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

// ---------------------------------------------------------------- LoRA rank-r projection
// One warp per sorted row p (expert e = e(p)):  P[p, j] = s * <In[p, :], Wt[e, j, :]>.
template <int RP>
__global__ void lora_project_kernel(const uint4* __restrict__ In, int vpr, const uint4* __restrict__ Wt, int r,
                                    float scale, const int32_t* __restrict__ offsets, int E, int64_t N,
                                    bf16* __restrict__ P) {
    extern __shared__ int32_t offs[];
    for (int i = threadIdx.x; i <= E; i += blockDim.x) offs[i] = offsets[i];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t p = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < N; p += nwarps) {
        const int e = expert_of_row(offs, E, (int)p);
        float acc[RP];
#pragma unroll
        for (int j = 0; j < RP; ++j) acc[j] = 0.f;
        const uint4* in = In + p * vpr;
        const uint4* w = Wt + (int64_t)e * r * vpr;
        for (int v = lane; v < vpr; v += 32) {
            float a[8];
            unpack8(__ldg(in + v), a);
#pragma unroll
            for (int j = 0; j < RP; ++j) {
                if (j < r) {
                    float b[8];
                    unpack8(__ldg(w + (int64_t)j * vpr + v), b);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[j] = fmaf(a[i], b[i], acc[j]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < RP; ++j) {
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], d);
        }
#pragma unroll
        for (int j = 0; j < RP; ++j)
            if (lane == (j & 31)) P[p * RP + j] = f2bf(j < r ? scale * acc[j] : 0.f);
    }
}

cudaError_t launch_lora_project(const void* In, int K, const void* Wt, int r, int rp, float scale,
                                const int32_t* offsets, int E, int64_t N, void* P, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>((N + 7) / 8, (int64_t)num_sms() * 8);
    const size_t smem = (size_t)(E + 1) * sizeof(int32_t);
    const uint4* in = (const uint4*)In;
    const uint4* wt = (const uint4*)Wt;
    if (rp == 16)
        lora_project_kernel<16><<<(unsigned)blocks, threads, smem, s>>>(in, K / 8, wt, r, scale, offsets, E, N, (bf16*)P);
    else if (rp == 32)
        lora_project_kernel<32><<<(unsigned)blocks, threads, smem, s>>>(in, K / 8, wt, r, scale, offsets, E, N, (bf16*)P);
    else
        lora_project_kernel<64><<<(unsigned)blocks, threads, smem, s>>>(in, K / 8, wt, r, scale, offsets, E, N, (bf16*)P);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- LoRA weight gradients
// D[e, j, m] = sum_{p in expert e} Small[p, j] * Big[p, m], rows visited in ascending
// order by one thread per column m (deterministic).  Experts without rows get zeros.
template <int RP>
__global__ void lora_wgrad_kernel(const bf16* __restrict__ Small, int r, const bf16* __restrict__ Big, int M,
                                  const int32_t* __restrict__ offsets, bf16* __restrict__ D) {
    constexpr int kRows = 32;
    __shared__ float sm[kRows][RP];
    const int e = blockIdx.y;
    const int m = blockIdx.x * blockDim.x + threadIdx.x;
    const int beg = offsets[e], end = offsets[e + 1];
    float acc[RP];
#pragma unroll
    for (int j = 0; j < RP; ++j) acc[j] = 0.f;
    for (int p0 = beg; p0 < end; p0 += kRows) {
        const int nr = min(kRows, end - p0);
        __syncthreads();
        for (int i = threadIdx.x; i < kRows * RP; i += blockDim.x) {
            const int rr = i / RP, j = i % RP;
            sm[rr][j] = rr < nr ? bf2f(Small[(int64_t)(p0 + rr) * RP + j]) : 0.f;
        }
        __syncthreads();
        if (m < M) {
            for (int rr = 0; rr < nr; ++rr) {
                const float b = bf2f(Big[(int64_t)(p0 + rr) * M + m]);
#pragma unroll
                for (int j = 0; j < RP; ++j) acc[j] = fmaf(sm[rr][j], b, acc[j]);
            }
        }
    }
    if (m < M) {
#pragma unroll
        for (int j = 0; j < RP; ++j)
            if (j < r) D[((int64_t)e * r + j) * M + m] = f2bf(acc[j]);
    }
}

size_t lora_wgrad_partial_elems(int64_t, int, int, int) { return 0; }

cudaError_t launch_lora_wgrad(const void* Small, int rp, int r, const void* Big, int M,
                              const int32_t* offsets, int E, int64_t, void* D, float*, size_t,
                              cudaStream_t s) {
    const int threads = 256;
    dim3 grid((M + threads - 1) / threads, E);
    if (rp == 16)
        lora_wgrad_kernel<16><<<grid, threads, 0, s>>>((const bf16*)Small, r, (const bf16*)Big, M, offsets, (bf16*)D);
    else if (rp == 32)
        lora_wgrad_kernel<32><<<grid, threads, 0, s>>>((const bf16*)Small, r, (const bf16*)Big, M, offsets, (bf16*)D);
    else
        lora_wgrad_kernel<64><<<grid, threads, 0, s>>>((const bf16*)Small, r, (const bf16*)Big, M, offsets, (bf16*)D);
    return cudaGetLastError();
}

}  // namespace moe
