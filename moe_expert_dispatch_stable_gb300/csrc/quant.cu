// FP8 (e4m3) expert base weights: per matrix and column, a power-of-two scale
// 2^ceil(log2(amax / 448)) and e4m3 codes rounded to nearest even.  With a
// power-of-two scale the division is exact and every dequantised value
// code * scale is a bf16 value (exactly, unless the scale is so small that it falls
// below bf16's normal range and rounds there), so the quantised base weights are
// themselves a set of bf16 weights (QLoRA-style frozen low-precision base,
// the pages' QLoRA variant of the expert layer, in the FP8 format).
//
// NF4 (4-bit NormalFloat) expert base weights: QLoRA's data type, the pages' "QLoRA
// 4-bit" base.  16 code values (normal quantiles normalised to [-1, 1]), one float32
// absmax per 64 consecutive elements of a row (stored block-major, [m][block][row], so
// that the GEMM's TMA fetches a stage's scales as one contiguous run), nearest code, two
// codes per byte; the dequantised weight is bf16(T[code] * absmax), formed inside the GEMM
// pipeline.
#include "common.cuh"
#include "kernels.h"

#include <cuda_fp8.h>

#include <algorithm>
#include <cmath>

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

// ---------------------------------------------------------------- NF4
namespace {

double normal_cdf(double x) { return 0.5 * std::erfc(-x / std::sqrt(2.0)); }

// inverse of the standard normal CDF on (1/2, 1), by bisection on normal_cdf
double normal_quantile(double p) {
    double lo = 0.0, hi = 8.0;
    for (int i = 0; i < 200; ++i) {
        const double mid = 0.5 * (lo + hi);
        if (normal_cdf(mid) < p) lo = mid;
        else hi = mid;
    }
    return 0.5 * (lo + hi);
}

// probability `i` steps of (1/2 - delta) / n from delta; the product is kept out of the sum
// so that no compiler fuses the two roundings into one
double nf4_probability(double delta, int i, int n) {
    const double step = (0.5 - delta) / n;
    volatile double offset = i * step;
    return delta + offset;
}

}  // namespace

// The QLoRA NormalFloat construction: quantiles of N(0, 1) at probabilities evenly spaced
// from delta towards 1/2 (8 for the positive values, 7 for the negative ones, mirrored),
// an exact zero, delta = 1 - (1/32 + 1/30) / 2 so that the outermost quantile is finite;
// divided by the largest and rounded to float32.  Code i is the i-th smallest value.
const Nf4Table& nf4_table() {
    static const Nf4Table table = [] {
        const double delta = 1.0 - 0.5 * (1.0 / 32.0 + 1.0 / 30.0);
        double v[16];
        int n = 0;
        for (int i = 0; i < 7; ++i) v[n++] = -normal_quantile(nf4_probability(delta, i, 7));
        v[n++] = 0.0;
        for (int i = 7; i >= 0; --i) v[n++] = normal_quantile(nf4_probability(delta, i, 8));
        Nf4Table t;
        for (int i = 0; i < 16; ++i) t.v[i] = (float)(v[i] / v[15]);
        return t;
    }();
    return table;
}

// nearest code value to w / a in float32, the lower code on a tie; code 7 (the zero) when
// the block is all zero
__device__ __forceinline__ uint32_t nf4_code(float w, float a, const Nf4Table& T) {
    if (!(a > 0.f)) return 7u;
    const float x = __fdiv_rn(w, a);
    uint32_t best = 0;
    float bd = fabsf(__fsub_rn(x, T.v[0]));
#pragma unroll
    for (int c = 1; c < 16; ++c) {
        const float d = fabsf(__fsub_rn(x, T.v[c]));
        if (d < bd) {
            bd = d;
            best = (uint32_t)c;
        }
    }
    return best;
}

// One warp per block of 64 elements (grid-stride); lane l holds elements 2l and 2l+1 and
// writes their byte.  Rows are a whole number of blocks, so block b of the flat weight
// array is (matrix m, row r, column block c) with b = (m * rows + r) * nblk + c, and its
// codes sit at the same flat index; its scale goes to absmax[m][c][r].
__global__ void quantize_nf4_kernel(const bf16* __restrict__ W, int64_t n_blocks, int64_t rows, int nblk,
                                    uint8_t* __restrict__ Wq, float* __restrict__ absmax, const Nf4Table T) {
    const int lane = threadIdx.x & 31;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t stride = (int64_t)gridDim.x * wpb;
    for (int64_t b = blockIdx.x * wpb + (threadIdx.x >> 5); b < n_blocks; b += stride) {
        const float2 w = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(W + b * 64)[lane]);
        float a = fmaxf(fabsf(w.x), fabsf(w.y));
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, d));
        Wq[b * 32 + lane] = (uint8_t)(nf4_code(w.x, a, T) | (nf4_code(w.y, a, T) << 4));
        if (lane == 0) {
            const int64_t c = b % nblk, mr = b / nblk;                 // mr = m * rows + r
            const int64_t m = mr / rows, r = mr % rows;
            absmax[(m * nblk + c) * rows + r] = a;
        }
    }
}

cudaError_t launch_quantize_nf4(const void* W, int64_t n_mat, int64_t rows, int cols, void* Wq, float* absmax,
                                cudaStream_t s) {
    if (cols % 64 != 0) return cudaErrorInvalidValue;
    const int64_t n_blocks = n_mat * rows * (cols / 64);
    if (n_blocks == 0) return cudaSuccess;
    const int grid = (int)std::min<int64_t>((n_blocks + 7) / 8, 16384);
    quantize_nf4_kernel<<<grid, 256, 0, s>>>((const bf16*)W, n_blocks, rows, cols / 64, (uint8_t*)Wq, absmax,
                                             nf4_table());
    return cudaGetLastError();
}

}  // namespace moe
