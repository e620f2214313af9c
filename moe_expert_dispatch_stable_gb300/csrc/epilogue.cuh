// Epilogue arithmetic of the grouped GEMMs (shared by both GEMM engines).
//
// SwiGLU (named among Unsloth's hand-written kernels in the GPU MODE lecture 32
// notes; read as h = silu(g) * u with g the first I and u the last I columns
// of the gate_up product) and its hand-derived derivative:
//   dh/dg = u * sig(g) * (1 + g (1 - sig(g))),  dh/du = silu(g) = g sig(g).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {

__device__ __forceinline__ float swiglu_f(float g, float u) { return g * sigmoidf_(g) * u; }

__device__ __forceinline__ void dswiglu_f(float dh, float g, float u, float& dg, float& du) {
    const float sg = sigmoidf_(g);
    dg = dh * u * sg * (1.0f + g * (1.0f - sg));
    du = dh * g * sg;
}

// Scalar epilogue: row p (sorted order), logical column n.
template <int EPI>
__device__ __forceinline__ void epilogue_store(const GroupedGemm& g, int p, int n, float acc, float acc2) {
    if constexpr (EPI == EPI_SWIGLU) {
        const int I = g.Ncols;
        bf16* GU = (bf16*)g.out0;
        bf16* h = (bf16*)g.out1;
        GU[(int64_t)p * 2 * I + n] = f2bf(acc);
        GU[(int64_t)p * 2 * I + I + n] = f2bf(acc2);
        h[(int64_t)p * I + n] = f2bf(swiglu_f(acc, acc2));
    } else if constexpr (EPI == EPI_ROWSCALE_F32) {
        ((float*)g.out0)[(int64_t)p * g.ldo + n] = g.w_sorted[p] * acc;
    } else if constexpr (EPI == EPI_DSWIGLU) {
        const int I = g.Ncols;
        const bf16* GU = (const bf16*)g.gu_in;
        const float gg = bf2f(GU[(int64_t)p * 2 * I + n]);
        const float uu = bf2f(GU[(int64_t)p * 2 * I + I + n]);
        float dg, du;
        dswiglu_f(acc, gg, uu, dg, du);
        bf16* dGU = (bf16*)g.out0;
        dGU[(int64_t)p * 2 * I + n] = f2bf(dg);
        dGU[(int64_t)p * 2 * I + I + n] = f2bf(du);
    } else {
        ((float*)g.out0)[(int64_t)p * g.ldo + n] = acc;
    }
}

}  // namespace moe
