// Row kernels of the MoE-LoRA layer: the permuted-row gather (with the
// routing-weight scale and the routing-weight gradient for the backward) and
// the deterministic, routing-weighted per-token combine.  Both are HBM-bound,
// with a couple of flops per element.
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

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
// output of the slot), accumulated in fp32 while the row is in registers.  Used for
// that gradient and for rows that are not a multiple of 16 columns; every other
// gather takes the chunked kernel below.
__global__ void gather_rows_kernel(const uint4* __restrict__ src, int vpr, const int32_t* __restrict__ perm,
                                   const float* __restrict__ w_sorted, int64_t N, int k,
                                   uint4* __restrict__ dst, const uint4* __restrict__ O, float* __restrict__ d_w,
                                   int32_t* status) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t p = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < N; p += nwarps) {
        const int slot = perm[p];
        if (!dbg_index_ok(slot, N, status)) continue;
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

// Gather without the weight gradient (the forward's x -> x_perm, the backward's weighted
// dy -> dY_perm): one warp per (sorted row, chunk of 32 * kUpl 32-byte units), each lane
// issuing all its 32-byte loads before its stores.  Rows are 32-byte aligned (H % 16 == 0,
// 32-byte aligned buffers).  With w_sorted, every element is scaled by the row's routing
// weight (fp32 product, rounded to bf16), the same arithmetic as the one-warp-per-row kernel.
constexpr int kUpl = 4;

__global__ void gather_rows32_kernel(const uint8_t* __restrict__ src, int units, const int32_t* __restrict__ perm,
                                     const float* __restrict__ w_sorted, int64_t N, int k,
                                     uint8_t* __restrict__ dst, int32_t* status) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int cpr = (units + 32 * kUpl - 1) / (32 * kUpl);
    const int64_t tasks = N * cpr;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t row_bytes = (int64_t)units * 32;
    for (int64_t task = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; task < tasks; task += nwarps) {
        const int64_t p = task / cpr;
        const int c = (int)(task - p * cpr);
        const int64_t slot = perm[p];
        if (!dbg_index_ok(slot, N, status)) continue;
        const int64_t t = slot / k;
        const float w = w_sorted != nullptr ? w_sorted[p] : 1.0f;
        const uint8_t* s = src + t * row_bytes;
        uint8_t* d = dst + p * row_bytes;
        uint4 a[kUpl], b[kUpl];
#pragma unroll
        for (int i = 0; i < kUpl; ++i) {
            const int u = (c * kUpl + i) * 32 + lane;
            if (u < units) tc::ld32_nc(s + (int64_t)u * 32, a[i], b[i]);
        }
#pragma unroll
        for (int i = 0; i < kUpl; ++i) {
            const int u = (c * kUpl + i) * 32 + lane;
            if (u < units) {
                if (w_sorted != nullptr) {
                    float f[16];
                    unpack8(a[i], f);
                    unpack8(b[i], f + 8);
#pragma unroll
                    for (int q = 0; q < 16; ++q) f[q] *= w;
                    a[i] = pack8(f);
                    b[i] = pack8(f + 8);
                }
                tc::st32(d + (int64_t)u * 32, a[i], b[i]);
            }
        }
    }
}

cudaError_t launch_gather_rows(const void* src, int H, const int32_t* perm, const float* w_sorted,
                               int64_t N, int k, void* dst, const void* O, float* d_w, int32_t* status,
                               cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    const int threads = 256;
    if (d_w == nullptr && H % 16 == 0) {
        const int units = H / 16;
        const int64_t tasks = N * ((units + 32 * kUpl - 1) / (32 * kUpl));
        const int64_t blocks = std::min<int64_t>((tasks + 7) / 8, (int64_t)num_sms() * 16);
        return launch_pdl(gather_rows32_kernel, dim3((unsigned)blocks), dim3(threads), 0, s, (const uint8_t*)src,
                          units, perm, w_sorted, N, k, (uint8_t*)dst, status);
    }
    const int64_t blocks = std::min<int64_t>((N + 7) / 8, (int64_t)num_sms() * 16);
    return launch_pdl(gather_rows_kernel, dim3((unsigned)blocks), dim3(threads), 0, s, (const uint4*)src, H / 8, perm,
                      w_sorted, N, k, (uint4*)dst, (const uint4*)O, d_w, status);
}

// ---------------------------------------------------------------- combine
// out[t] = sum_{j=0}^{k-1} w_j * src[inv_perm[t*k+j]] in that order, summed in fp32.
// One warp per (token, chunk of 32 * combine_upl units of 16 columns); each lane loads the k
// slots' 16 columns with one 32-byte access per slot (the slot rows are bf16: the forward's
// expert outputs O and the backward's per-slot input gradients).
template <typename SrcT>
__device__ __forceinline__ void load16(const SrcT* row, int u, float* a);

template <>
__device__ __forceinline__ void load16<bf16>(const bf16* row, int u, float* a) {
    uint4 x, y;
    tc::ld32_cs(row + (int64_t)u * 16, x, y);
    unpack8(x, a);
    unpack8(y, a + 8);
}

// units per lane and task (measured: one keeps the most warps resident)
template <typename SrcT>
__host__ __device__ constexpr int combine_upl() { return 1; }

template <typename SrcT>
__global__ void combine_kernel(const SrcT* __restrict__ src, const float* __restrict__ w_sorted,
                               const int32_t* __restrict__ inv_perm, int64_t T, int k, int H,
                               bf16* __restrict__ out, int32_t* status) {
    pdl_wait();
    pdl_trigger();
    constexpr int kC = combine_upl<SrcT>();
    const int lane = threadIdx.x & 31;
    const int units = H / 16;
    const int cpr = (units + 32 * kC - 1) / (32 * kC);
    const int64_t tasks = T * cpr;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t task = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; task < tasks; task += nwarps) {
        const int64_t t = task / cpr;
        const int c = (int)(task - t * cpr);
        float acc[kC][16];
#pragma unroll
        for (int i = 0; i < kC; ++i)
#pragma unroll
            for (int q = 0; q < 16; ++q) acc[i][q] = 0.f;
        // the slots' rows and weights, 32 at a time one per lane, broadcast in slot order
        for (int j0 = 0; j0 < k; j0 += 32) {
            const int kj = min(32, k - j0);
            int64_t my_row = lane < kj ? inv_perm[t * k + j0 + lane] : 0;
            const bool my_ok = lane >= kj || dbg_index_ok(my_row, T * k, status);
            if (!my_ok) my_row = 0;                         // debug build: a bad row adds nothing
            const float my_w = !my_ok ? 0.0f : ((lane < kj && w_sorted != nullptr) ? w_sorted[my_row] : 1.0f);
#pragma unroll 4
            for (int j = 0; j < kj; ++j) {
                const int64_t row = __shfl_sync(0xffffffffu, my_row, j);
                const float w = __shfl_sync(0xffffffffu, my_w, j);
#pragma unroll
                for (int i = 0; i < kC; ++i) {
                    const int u = (c * kC + i) * 32 + lane;
                    if (u < units) {
                        float a[16];
                        load16<SrcT>(src + row * H, u, a);
#pragma unroll
                        for (int q = 0; q < 16; ++q) acc[i][q] = fmaf(w, a[q], acc[i][q]);
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kC; ++i) {
            const int u = (c * kC + i) * 32 + lane;
            if (u < units) tc::st32(out + t * H + (int64_t)u * 16, pack8(acc[i]), pack8(acc[i] + 8));
        }
    }
}

// ---------------------------------------------------------------- SwiGLU rows
// h[p] = SwiGLU(GU[p]) for every sorted row, 8 columns per thread and step: the forward's
// h rebuilt from the saved bf16 GU.  The gate_up epilogue forms h from the same bf16 gate
// and up values with the same arithmetic (swiglu_f, round to nearest bf16), so the rows
// are bit-identical to the ones it stored.
__global__ void swiglu_rows_kernel(const uint4* __restrict__ gu, int i8, int64_t N, uint4* __restrict__ h) {
    pdl_wait();
    pdl_trigger();
    const int64_t units = N * i8;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += step) {
        const int64_t p = u / i8;
        const int c = (int)(u - p * i8);
        float g[8], v[8], o[8];
        unpack8(__ldg(gu + p * 2 * i8 + c), g);
        unpack8(__ldg(gu + p * 2 * i8 + i8 + c), v);
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] = swiglu_f(g[j], v[j]);
        h[p * i8 + c] = pack8(o);
    }
}

cudaError_t launch_swiglu_rows(const void* gu, int I, int64_t N, void* h, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    if (I % 8 != 0) return cudaErrorInvalidValue;
    const int threads = 256;
    const int64_t units = N * (I / 8);
    const int64_t blocks = std::min<int64_t>((units + threads - 1) / threads, (int64_t)num_sms() * 16);
    return launch_pdl(swiglu_rows_kernel, dim3((unsigned)blocks), dim3(threads), 0, s, (const uint4*)gu, I / 8, N,
                      (uint4*)h);
}

cudaError_t launch_combine(const void* src, const float* w_sorted, const int32_t* inv_perm, int64_t T, int k, int H,
                           void* out, int32_t* status, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (H % 16 != 0) return cudaErrorInvalidValue;
    const int threads = 256;
    const int units = H / 16;
    const int upl = combine_upl<bf16>();
    const int64_t tasks = T * ((units + 32 * upl - 1) / (32 * upl));
    const int64_t blocks = std::min<int64_t>((tasks + 7) / 8, (int64_t)num_sms() * 16);
    return launch_pdl(combine_kernel<bf16>, dim3((unsigned)blocks), dim3(threads), 0, s, (const bf16*)src, w_sorted,
                      inv_perm, T, k, H, (bf16*)out, status);
}

}  // namespace moe
