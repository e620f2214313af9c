// FP8 (e4m3) expert base weights: per matrix and column, a power-of-two scale
// 2^ceil(log2(amax / 448)) and e4m3 codes rounded to nearest even.  With a
// power-of-two scale the division is exact and every dequantised value
// code * scale is a bf16 value (exactly, unless the scale is so small that it falls
// below bf16's normal range and rounds there), so the quantised base weights are
// themselves a set of bf16 weights (QLoRA-style frozen low-precision base,
// the pages' QLoRA variant of the expert layer, in the FP8 format).
#include "common.cuh"
#include "kernels.h"

#include <cuda_fp8.h>

namespace moe {

// Smallest e with amax <= 448 * 2^e, by exact comparisons (0 for an all-zero column).
__device__ __forceinline__ int pow2_exponent(float amax) {
    if (!(amax > 0.f)) return 0;
    int e = ilogbf(amax) - 8;                     // 448 = 1.75 * 2^8
    while (amax > ldexpf(448.0f, e)) ++e;
    while (amax <= ldexpf(448.0f, e - 1)) --e;
    return e;
}

// grid (ceil(cols / 256), n_mat), one thread per column.
__global__ void quantize_fp8_kernel(const bf16* __restrict__ W, int64_t rows, int cols, uint8_t* __restrict__ Wq,
                                    float* __restrict__ scale) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t m = blockIdx.y;
    if (c >= cols) return;
    const bf16* w = W + m * rows * cols + c;
    float amax = 0.f;
    for (int64_t r = 0; r < rows; ++r) amax = fmaxf(amax, fabsf(bf2f(w[r * cols])));
    const int e = pow2_exponent(amax);
    scale[m * cols + c] = ldexpf(1.0f, e);         // may be an fp32 subnormal for tiny columns
    uint8_t* q = Wq + m * rows * cols + c;
    // w * 2^-e by exponent arithmetic: exact, and no reciprocal of a subnormal scale
    for (int64_t r = 0; r < rows; ++r)
        q[r * cols] = (uint8_t)__nv_cvt_float_to_fp8(ldexpf(bf2f(w[r * cols]), -e), __NV_SATFINITE, __NV_E4M3);
}

cudaError_t launch_quantize_fp8(const void* W, int64_t n_mat, int64_t rows, int cols, void* Wq, float* scale,
                                cudaStream_t s) {
    if (n_mat == 0 || rows == 0 || cols == 0) return cudaSuccess;
    dim3 grid((cols + 255) / 256, (unsigned)n_mat);
    quantize_fp8_kernel<<<grid, 256, 0, s>>>((const bf16*)W, rows, cols, (uint8_t*)Wq, scale);
    return cudaGetLastError();
}

}  // namespace moe
