// Internal launch interface between the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_lora.h"

namespace moe {

// ---- diagnostics (api.cu)
// Wait limit and forced stall of the next single-CTA tensor-core launch (a grouped GEMM on
// single-CTA tiles, a rank-r projection or a LoRA reduction): the library's full limit and
// no stall, unless moe_diag_force_timeout chose this launch.  Counts the launch.
struct DiagWait {
    uint64_t limit_ns;
    bool stall;
};
DiagWait diag_next_single_cta_launch();

// ---- routing (route.cu)
size_t route_workspace_bytes(int64_t N, int E);
cudaError_t launch_route(const void* idx, int idx_bytes, const float* topk_w, int64_t N, int E,
                         const moe_routing& out, void* ws, int32_t* dev_status, cudaStream_t s);
// Device address of the fixed MOE_ROUTE_STATIC_SCRATCH_BYTES scratch array (looked up once per device).
cudaError_t route_static_scratch(void** ptr);

// ---- row kernels (rowops.cu)
// dst[p, :] = src[perm[p] / k, :]   (optionally scaled by w_sorted[p], rounded to bf16).
// With O and d_w given: d_w[perm[p]] = <src[perm[p] / k, :], O[p, :]> (fp32), in the same pass.
// `status` (may be null): the debug build's MOE_DEV_BAD_INDEX for a perm entry outside [0, N).
cudaError_t launch_gather_rows(const void* src, int H, const int32_t* perm, const float* w_sorted,
                               int64_t N, int k, void* dst, const void* O, float* d_w, int32_t* status,
                               cudaStream_t s);
// out[t, :] = bf16( sum_{j<k} w * src[inv_perm[t*k+j], :] ) over bf16 slot rows, w = w_sorted[inv_perm[t*k+j]]
// (or 1 when w_sorted is null), fp32 sum in the fixed order j = 0..k-1
cudaError_t launch_combine(const void* src, const float* w_sorted, const int32_t* inv_perm, int64_t T, int k, int H,
                           void* out, int32_t* status, cudaStream_t s);
// h [N, I] = SwiGLU of GU [N, 2I] row by row (bf16 in and out)
cudaError_t launch_swiglu_rows(const void* gu, int I, int64_t N, void* h, cudaStream_t s);

// ---- FP8 expert weights (quant.cu)
// scale[m, c] = 2^ceil(log2(amax_r |W[m, r, c]| / 448)), Wq[m, r, c] = e4m3_rn(W[m, r, c] / scale[m, c])
cudaError_t launch_quantize_fp8(const void* W, int64_t n_mat, int64_t rows, int cols, void* Wq, float* scale,
                                cudaStream_t s);

// ---- NF4 (4-bit NormalFloat) expert weights (quant.cu)
// The 16 NF4 code values, ascending, computed once on the host from their definition
// (normal quantiles at evenly spaced probabilities, normalised to [-1, 1]).
struct Nf4Table {
    float v[16];
};
const Nf4Table& nf4_table();
// Per 64 consecutive elements of a row: absmax[m, b, r] = max |W[m, r, 64b .. 64b+63]|
// (block-major: the scales of one column block are contiguous over the rows); each
// element's code is the nearest table value to W / absmax (float32, ties to the lower code;
// code 7 when the block is all zero); Wq packs two codes per byte, the even column in the
// low nibble.  cols % 64 == 0.
cudaError_t launch_quantize_nf4(const void* W, int64_t n_mat, int64_t rows, int cols, void* Wq, float* absmax,
                                cudaStream_t s);

// ---- router (router.cu)
cudaError_t launch_router_topk(const float* logits, int64_t T, int E, int k, int32_t* topk_idx, float* topk_w,
                               cudaStream_t s);
cudaError_t launch_router_bwd(const float* logits, const int32_t* topk_idx, const float* d_topk_w, int64_t T, int E,
                              int k, float* d_logits, cudaStream_t s);

// ---- packed-sequence metadata (packed.cu)
// One CTA: a token starts a sample when it is token 0 or position_ids[t] == 0;
// cu_seqlens[0..n] = the samples' first tokens then T, seq_id[t] = the token's sample,
// *n_seqs = n, *max_seqlen = the longest sample.  T <= 2^30.
cudaError_t launch_packed_metadata(const void* position_ids, int pos_bytes, int64_t T, int32_t* cu_seqlens,
                                   int32_t* seq_id, int32_t* n_seqs, int32_t* max_seqlen, cudaStream_t s);
// mask[i * T + j] = (cu_seqlens[seq_id[i]] <= j <= i), uint8 [T, T] row-major; mask 16-byte aligned.
cudaError_t launch_packed_mask(const int32_t* cu_seqlens, const int32_t* seq_id, int64_t T, uint8_t* mask,
                               cudaStream_t s);

// ---- per-expert LoRA weight gradients (gemm_wgrad.cu)
// D[e, j, m] = sum_{p in rows of e} Small[p, j] * Big[p, m]  (bf16 out [E, r, M]) on the
// tensor cores, one CTA per (problem, expert, 128 columns), fixed row order, zeros for
// empty experts.  One or two problems (same experts, same rank) per launch.
struct WgradProblem {
    const void* Small;   // [N, RP] bf16
    const void* Big;     // [N, M] bf16
    int M;
    void* D;             // [E, r, M] bf16
};
cudaError_t launch_lora_wgrad_tc(const WgradProblem* probs, int nprob, int rp, int r, const int32_t* offsets, int E,
                                 int64_t N, int32_t* dev_status, cudaStream_t s);

// ---- grouped GEMMs (gemm_tc.cu)
enum GemmEpi : int {
    EPI_SWIGLU = 0,     // paired gate/up accumulators -> GU (bf16, [N,2I]) and h (bf16, [N,I])
    EPI_BF16 = 1,       // out_bf16[p, n] = acc
    EPI_DSWIGLU = 2,    // acc = dh; reads GU, writes dGU (bf16 [N,2I])
    EPI_PROJ = 4        // out_bf16[p, 0:Ncols] = scale * acc  (rank-r projection, Ncols = RP)
};

struct GroupedGemm {
    // problem: for every expert e and sorted row p in [offsets[e], offsets[e+1]):
    //   acc[p, n] = sum_c A[p, c] B_e(c, n) + sum_j A2[p, j] B2_e(j, n),  n < Ncols
    // (for EPI_SWIGLU a second accumulator uses B columns n + Ncols: the "up" half)
    int64_t N;            // total sorted rows
    int E;
    int K;                // contraction length of the main product
    int Ncols;            // logical output columns
    const void* A;        // [N, K] bf16, K contiguous
    const void* B;        // bf16 expert stack
    bool b_mn_major;      // true: B_e(c, n) = B[e][c][n] (row length ldb); false: B[e][n][c]
    int b_quant;          // 0: bf16 B; 8: e4m3 codes, value = code * b_scale[e * ldb + column of B[e]];
                          // 4: NF4 codes, two per byte, value = bf16(T[code] * b_scale[block]), one
                          //    scale per 64 consecutive elements of a row of B[e], stored
                          //    [E][ldb / 64][rows of B[e]]
    const float* b_scale; // the scales of a quantised B
    int ldb;              // elements per row of B[e]
    int64_t b_expert_stride;  // elements between experts
    const void* A2;       // [N, RP] bf16 (LoRA rank activations, pre-scaled by s), or null
    int rp;               // row length of A2
    int r;                // contraction length of the LoRA product
    const void* B2;       // [E][r][ldb2] bf16 (MN-major), or null
    int ldb2;
    int64_t b2_expert_stride;
    const int32_t* offsets;      // [E+1]
    const int32_t* tile_offsets; // [E+1], 128-row tiles
    const void* gu_in;           // EPI_DSWIGLU: GU [N, 2*Ncols]
    void* out0;                  // EPI_SWIGLU: GU; EPI_DSWIGLU: dGU; BF16: bf16 out
    void* out1;                  // EPI_SWIGLU: h
    int ldo;                     // row length of the BF16 output
    float scale;                 // EPI_PROJ
    int h_from_gu;               // EPI_SWIGLU: h from the bf16-rounded gate / up values (as stored)
    int epi;
    int32_t* dev_status;
};

// Product engine (tcgen05 / TMEM / TMA persistent kernel).
cudaError_t launch_grouped_gemm(const GroupedGemm& g, cudaStream_t s);


}  // namespace moe
