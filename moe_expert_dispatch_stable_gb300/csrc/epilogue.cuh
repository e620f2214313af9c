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

}  // namespace moe
