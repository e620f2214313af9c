/*
 * moe_lora.h -- C ABI of the GB300 (sm_103a) MoE-LoRA expert layer.
 *
 * Three operations, all enqueued on the caller's CUDA stream, none of which
 * synchronises with the host or copies anything back to it:
 *
 *   moe_route     group the T*k routed slots by expert (histogram, exclusive
 *                 scan to offsets, stable scatter).
 *   moe_lora_fwd  y = sum_j w[t,j] * SwiGLU-expert_{e(t,j)}(x[t]) with
 *                 Split-LoRA on both projections.
 *   moe_lora_bwd  dx and the per-expert LoRA gradients dA_gu, dB_gu, dA_d,
 *                 dB_d for L = <dy, y> (the base weights are frozen).
 *
 * Sources.  Routing: the blog post on Unsloth x NVIDIA training speed-ups
 * (d9249.github.io, section "core idea / structure / how it works", GPT-OSS MoE
 * routing paragraphs): flatten the top-k assignment, stable-sort by expert id,
 * bincount once, slice by offsets, instead of one torch.where query per
 * expert.  Grouped matmul and Split-LoRA: the Unsloth 2026 wiki page on GRPO,
 * MoE and memory-efficient fine-tuning, section "Optimisation 3: grouped_mm and
 * Split-LoRA for MoE training": all experts' weights stacked in one tensor,
 * group sizes equal to the routing counts, and the LoRA product applied after
 * the base product (x W + s (x A) B) instead of materialising W + BA.
 *
 * Conventions for every function:
 *  - All tensors are dense row-major; bf16 tensors are passed as uint16_t*.
 *  - Every pointer is a DEVICE pointer unless stated otherwise, 16-byte aligned,
 *    owned by the caller; the activation buffers x, y, dy, dx, saved and the
 *    workspaces of moe_lora_fwd / moe_lora_bwd (and their _fp8 / _nf4 forms) are 32-byte
 *    aligned (their rows are moved with 32-byte accesses).  Buffers whose size is a multiple of T (x, y, dy, dx,
 *    perm, inv_perm, w_sorted, saved, workspaces) may be NULL when T == 0.  The library allocates no device memory and keeps no
 *    state beyond a per-device cache of the SM count and of a driver entry point.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *  - A non-zero return is a host-side error found before anything was enqueued
 *    (bad argument, unsupported size, workspace too small) or a CUDA launch
 *    error; nothing is launched in the first three cases.
 *  - Errors only the device can see are OR-ed into *dev_status (a device int32
 *    the caller zeroes and reads when it wants): MOE_DEV_BAD_EXPERT_ID for an
 *    expert id outside [0, E), MOE_DEV_TIMEOUT when a bounded wait inside a
 *    kernel gave up.  When a bit is set the outputs are unspecified.
 *  - No function blocks the host.  moe_route, moe_lora_fwd, moe_lora_bwd (and the
 *    _fp8 / _nf4 forms) can be captured in a CUDA graph.
 *
 * Sizes supported: 1 <= k <= E <= 1024, H and I multiples of 64, 1 <= r <= 64,
 * T >= 0 and T*k < 2^31.
 */
#ifndef MOE_LORA_H
#define MOE_LORA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t moe_status;

enum {
    MOE_OK = 0,
    MOE_ERR_NULL_ARG = 1,      /* a required pointer is NULL */
    MOE_ERR_BAD_DIMS = 2,      /* sizes outside the supported range */
    MOE_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte (activation buffers: 32-byte) aligned */
    MOE_ERR_WORKSPACE = 4,     /* workspace / saved buffer smaller than required */
    MOE_ERR_CUDA = 5,          /* a CUDA runtime / driver call failed */
    MOE_ERR_UNSUPPORTED = 6    /* device is not sm_103 or a needed driver entry point is missing */
};

enum {
    MOE_DEV_BAD_EXPERT_ID = 1,
    MOE_DEV_TIMEOUT = 2,
    /* Debug build of the library only (libmoe_lora_gb300_debug.so, compiled with
     * MOE_DEBUG=1): an index read from a routing buffer (perm, inv_perm, offsets,
     * tile_offsets) was out of range; the access was skipped.  The release build
     * does not check these indices: they must come from moe_route. */
    MOE_DEV_BAD_INDEX = 4
};

/* Row tile of the grouped GEMMs; tile_offsets counts tiles of this many rows. */
#define MOE_TILE_M 128

typedef struct moe_dims {
    int64_t T;      /* tokens */
    int32_t H;      /* hidden size (x, y rows) */
    int32_t I;      /* expert intermediate size (gate_up: H -> 2I, down: I -> H) */
    int32_t E;      /* number of experts */
    int32_t k;      /* experts per token */
    int32_t r;      /* LoRA rank */
    float scale;    /* LoRA scale s (alpha / r) */
} moe_dims;

/* Outputs of moe_route, inputs of moe_lora_fwd / moe_lora_bwd (device pointers). */
typedef struct moe_routing {
    int32_t* perm;          /* [T*k]  perm[p] = flat slot t*k+j at sorted position p */
    int32_t* inv_perm;      /* [T*k]  inv_perm[perm[p]] = p */
    int32_t* counts;        /* [E]    rows routed to each expert */
    int32_t* offsets;       /* [E+1]  exclusive prefix sum of counts */
    int32_t* tile_offsets;  /* [E+1]  exclusive prefix sum of ceil(counts / MOE_TILE_M) */
    float* w_sorted;        /* [T*k]  w_sorted[p] = topk_w_flat[perm[p]] (bit copy) */
} moe_routing;

/* ABI version of this header (bumped on any signature change). */
MOE_API int32_t moe_abi_version(void);

/* Static string for a status code. */
MOE_API const char* moe_status_string(moe_status s);

/* ---------------------------------------------------------------- routing
 * Bytes of device workspace moe_route needs for T tokens, k slots, E experts. */
MOE_API moe_status moe_route_workspace_size(int64_t T, int32_t k, int32_t E, size_t* bytes);

/* Group the routed slots by expert.
 *  topk_idx   [T, k] expert ids, int32 (idx_bytes = 4) or int64 (idx_bytes = 8)
 *  topk_w     [T, k] float32 routing weights (only copied, reordered)
 *  out        device pointers of the outputs (see moe_routing)
 * The order inside an expert is the ascending flat slot index t*k + j, i.e. a
 * stable sort of the flattened assignment by expert id.  Bit-exact and
 * deterministic.  An id outside [0, E) sets MOE_DEV_BAD_EXPERT_ID and that slot
 * is left out of every output.  Three stream operations: a 4-byte memset and
 * two kernels. */
MOE_API moe_status moe_route(const void* topk_idx, int32_t idx_bytes, const float* topk_w,
                     int64_t T, int32_t k, int32_t E, const moe_routing* out,
                     void* workspace, size_t workspace_bytes,
                     int32_t* dev_status, void* stream);

/* Routing for callers that cannot allocate device memory.
 *
 * No passage of the pages has a counterpart to this entry point: it exists for
 * callers of this library that cannot call cudaMalloc -- hosts whose device
 * memory is entirely owned by another allocator or a fixed pool (a framework's
 * caching allocator that must account for every byte, an embedded runtime with a
 * fixed arena), and latency-critical loops where an allocation could synchronise
 * the device.  Such a caller still passes every input and output, but no
 * workspace.
 *
 * It computes exactly what moe_route computes (same kernels, bit-identical
 * outputs); the routing scratch lives instead in one file-scope device array of
 * MOE_ROUTE_STATIC_SCRATCH_BYTES that every GPU loading the library holds until
 * the process exits.  The call needs moe_route_workspace_size(T, k, E) <=
 * MOE_ROUTE_STATIC_SCRATCH_BYTES; that size is exactly
 * align_up(ceil(T*k / 1024) * E * 4, 256) + 256 bytes (for example T*k <= 64512
 * slots at E = 1024, or T*k <= 523264 at E = 128).  Larger sizes return
 * MOE_ERR_WORKSPACE and launch nothing.
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and keeps it together with the device's current context; a
 * later call in a new context (after cudaDeviceReset, or a primary context
 * destroyed and made again) looks it up afresh.  Make the first call in a
 * context before any stream capture.  The call allocates nothing (no cudaMalloc, cudaFree or allocating
 * library routine) and clears the part of the array that must start at zero on
 * every call.  All calls share the array, so calls whose kernels overlap on the
 * GPU (several streams, or several host threads) race: serialise them. */
#define MOE_ROUTE_STATIC_SCRATCH_BYTES (256u * 1024u)
MOE_API moe_status moe_route_static(const void* topk_idx, int32_t idx_bytes, const float* topk_w,
                                    int64_t T, int32_t k, int32_t E, const moe_routing* out,
                                    int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------- forward
 * Bytes of the `saved` buffer (activations kept for the backward pass) and of
 * the forward workspace. */
MOE_API moe_status moe_lora_fwd_sizes(const moe_dims* d, size_t* saved_bytes, size_t* workspace_bytes);

/* Byte offsets inside `saved` of: x_perm [N,H], GU [N,2I], h [N,I],
 * XA_s [N,RP], HA_s [N,RP], O [N,H] (all bf16, N = T*k rows in sorted order,
 * RP = r rounded up to 16, 32 or 64, padding columns zero;
 * XA_s = s * x_perm A_gu^T, HA_s = s * h A_d^T, O = the unweighted expert
 * output of each slot).  For inspection and tests. */
MOE_API moe_status moe_lora_saved_layout(const moe_dims* d, size_t offsets[6], int32_t* rp);

/* Re-create the x_perm section of `saved` from the layer input x with the forward's
 * own gather (x_perm[p] = x[perm[p] / k]), bit-identical to what moe_lora_fwd wrote.
 * For a caller that keeps only the other sections between forward and backward (the
 * reload of offloaded activations in the blog post "Unsloth와 NVIDIA의 협업은 LLM 학습
 * 병목을 커널 밖에서 줄인다", section "핵심 아이디어 / 구조 / 동작 방식", moves GU .. HA_s back
 * and regathers x_perm instead of copying it).  x [T, H] bf16 (32-byte aligned), `rt`
 * the routing of the forward, `saved` as for moe_lora_fwd; nothing else in `saved` is
 * touched.  Asynchronous on `stream`. */
MOE_API moe_status moe_lora_saved_regather(const moe_dims* d, const moe_routing* rt, const uint16_t* x, void* saved,
                                           size_t saved_bytes, void* stream);

/* Re-create the h section of `saved` from its GU section: h = silu(g) * u row by row,
 * with g, u the stored bf16 values, fp32 arithmetic and round to nearest bf16.  That is
 * how moe_lora_fwd_h_from_gu forms h, so after that forward the result is bit-identical
 * to what it wrote (after moe_lora_fwd, whose h comes from the unrounded accumulators,
 * it is close but not identical).  For a caller that moves GU, XA_s and HA_s between
 * forward and backward but not h.  `saved` as for moe_lora_fwd; only h is written.
 * Asynchronous on `stream`. */
MOE_API moe_status moe_lora_saved_rebuild_h(const moe_dims* d, void* saved, size_t saved_bytes, void* stream);

/* Forward of the MoE-LoRA expert layer (Split-LoRA, SwiGLU, weighted combine).
 *  x     [T, H]                  W_gu [E, H, 2I] (gate = cols [0,I), up = [I,2I))
 *  A_gu  [E, r, H] (A^T, the PEFT lora_A layout)   B_gu [E, r, 2I]
 *  W_d   [E, I, H]   A_d [E, r, I]   B_d [E, r, H]
 *  y     [T, H] output, bf16
 * For every slot (t, j) with e = topk_idx[t, j]:
 *   GU = x[t] W_gu[e] + s (x[t] A_gu[e]^T) B_gu[e];  h = silu(GU[:I]) * GU[I:]
 *   (h from the fp32 accumulators; GU and h are then stored in bf16)
 *   o  = h W_d[e] + s (h A_d[e]^T) B_d[e];           y[t] = sum_j w[t,j] o_j
 * with bf16 operands, fp32 accumulation, and the k slots of a token summed in
 * the fixed order j = 0..k-1 (bitwise reproducible).  The forward needs no
 * workspace today (workspace_bytes is 0; `workspace` may be NULL). */
MOE_API moe_status moe_lora_fwd(const moe_dims* d, const moe_routing* rt,
                        const uint16_t* x,
                        const uint16_t* W_gu, const uint16_t* A_gu, const uint16_t* B_gu,
                        const uint16_t* W_d, const uint16_t* A_d, const uint16_t* B_d,
                        uint16_t* y,
                        void* saved, size_t saved_bytes,
                        void* workspace, size_t workspace_bytes,
                        int32_t* dev_status, void* stream);

/* moe_lora_fwd, except that h is formed from the gate and up values as stored (rounded
 * to bf16) instead of from the fp32 accumulators, so that moe_lora_saved_rebuild_h can
 * re-create h bit for bit from GU alone.  For a caller that offloads the saved
 * activations and moves h neither way; same arguments and sizes as moe_lora_fwd. */
MOE_API moe_status moe_lora_fwd_h_from_gu(const moe_dims* d, const moe_routing* rt, const uint16_t* x,
                                          const uint16_t* W_gu, const uint16_t* A_gu, const uint16_t* B_gu,
                                          const uint16_t* W_d, const uint16_t* A_d, const uint16_t* B_d, uint16_t* y,
                                          void* saved, size_t saved_bytes, void* workspace, size_t workspace_bytes,
                                          int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------- backward */
MOE_API moe_status moe_lora_bwd_workspace_size(const moe_dims* d, size_t* bytes);

/* Backward of moe_lora_fwd for L = <dy, y> with the base weights frozen.
 *  dy [T, H]; saved = the buffer moe_lora_fwd filled (same d, rt, weights).
 *  Outputs (bf16, same layouts as the parameters):
 *   dx [T, H], dA_gu [E, r, H], dB_gu [E, r, 2I], dA_d [E, r, I], dB_d [E, r, H]
 *  and, when d_topk_w is not NULL, the routing-weight gradient
 *   d_topk_w [T, k] float32: dL/dw[t,j] = <dy[t], expert_{e(t,j)}(x[t])>
 * Per slot: dO = w dy[t]; dh = dO W_d^T + s (dO B_d^T) A_d;
 *   dGU = SwiGLU'(GU) dh;  dx[t] += dGU W_gu^T + s (dGU B_gu^T) A_gu
 * Per expert (sums over its rows, fixed order, no float atomics):
 *   dA_d = s (dO B_d^T)^T h,  dB_d = s (h A_d^T)^T dO,
 *   dA_gu = s (dGU B_gu^T)^T x,  dB_gu = s (x A_gu^T)^T dGU.
 * Experts with no rows get exact zeros. */
MOE_API moe_status moe_lora_bwd(const moe_dims* d, const moe_routing* rt,
                        const uint16_t* dy,
                        const uint16_t* W_gu, const uint16_t* A_gu, const uint16_t* B_gu,
                        const uint16_t* W_d, const uint16_t* A_d, const uint16_t* B_d,
                        const void* saved, size_t saved_bytes,
                        uint16_t* dx, uint16_t* dA_gu, uint16_t* dB_gu,
                        uint16_t* dA_d, uint16_t* dB_d, float* d_topk_w,
                        void* workspace, size_t workspace_bytes,
                        int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------- FP8 expert base weights
 * A quantised frozen base (the pages' QLoRA variant of the expert layer, in the
 * FP8 e4m3 format): per matrix m and column c of W [n_mat, rows, cols] (bf16),
 *   scales[m, c] = 2^ceil(log2(max_r |W[m, r, c]| / 448))   (1 for an all-zero column)
 *   Wq[m, r, c]  = e4m3 code of W[m, r, c] / scales[m, c], round to nearest even.
 * With power-of-two scales the division is exact and every dequantised value
 * e4m3(Wq) * scale is exactly a bf16 number.  Wq uint8 [n_mat, rows, cols],
 * scales float32 [n_mat, cols].  One kernel; weight preparation, not the hot path. */
MOE_API moe_status moe_quantize_fp8(const uint16_t* W, int64_t n_mat, int64_t rows, int32_t cols,
                                    uint8_t* Wq, float* scales, void* stream);

/* moe_lora_fwd / moe_lora_bwd with FP8 base weights: Wq_gu [E, H, 2I] and Wq_d [E, I, H]
 * hold e4m3 codes with column scales s_gu [E, 2I] and s_d [E, H] (moe_quantize_fp8).
 * The GEMMs stream the codes (half the bytes of bf16) and dequantise them to bf16 in
 * shared memory before the tensor cores read them, so the results are bit-identical to
 * moe_lora_fwd / moe_lora_bwd called with the dequantised bf16 weights.  The LoRA
 * factors and activations stay bf16.  Same saved / workspace sizes.  The expert GEMMs
 * run on SM pairs (2-CTA clusters, each CTA dequantising half of a B tile); on a device
 * where no such cluster fits, the calls return MOE_ERR_CUDA. */
MOE_API moe_status moe_lora_fwd_fp8(const moe_dims* d, const moe_routing* rt, const uint16_t* x,
                                    const uint8_t* Wq_gu, const float* s_gu,
                                    const uint16_t* A_gu, const uint16_t* B_gu,
                                    const uint8_t* Wq_d, const float* s_d,
                                    const uint16_t* A_d, const uint16_t* B_d, uint16_t* y,
                                    void* saved, size_t saved_bytes,
                                    void* workspace, size_t workspace_bytes,
                                    int32_t* dev_status, void* stream);
MOE_API moe_status moe_lora_bwd_fp8(const moe_dims* d, const moe_routing* rt, const uint16_t* dy,
                                    const uint8_t* Wq_gu, const float* s_gu,
                                    const uint16_t* A_gu, const uint16_t* B_gu,
                                    const uint8_t* Wq_d, const float* s_d,
                                    const uint16_t* A_d, const uint16_t* B_d,
                                    const void* saved, size_t saved_bytes,
                                    uint16_t* dx, uint16_t* dA_gu, uint16_t* dB_gu,
                                    uint16_t* dA_d, uint16_t* dB_d, float* d_topk_w,
                                    void* workspace, size_t workspace_bytes,
                                    int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------- NF4 expert base weights
 * The pages' "QLoRA 4-bit" base (the Unsloth 2026 wiki page, section "supported models and
 * 2026 changes", model table; the GPU MODE lecture 32 notes, open questions, name QLoRA's
 * NF4), read as QLoRA's 4-bit NormalFloat data type.  Per matrix m, row r and block b of
 * 64 consecutive columns of W [n_mat, rows, cols] (bf16, cols a multiple of 64):
 *   absmax[m, b, r] = max |W[m, r, 64b .. 64b+63]|   (block-major: one column block's scales
 *                     are contiguous over the rows, so a GEMM stage fetches its scales as one
 *                     run with its codes)
 *   code of W[m, r, c] = the i in 0..15 whose T[i] is nearest to W[m, r, c] / absmax (both in
 *                        float32, the lower i on a tie; 7, the zero, when absmax is 0)
 *   Wq[m, r, c / 2]    = code(c even) | code(c odd) << 4
 * T = moe_nf4_codebook.  The dequantised weight is bf16(T[code] * absmax), the product in
 * float32 rounded to nearest even.  Wq uint8 [n_mat, rows, cols / 2], absmax float32
 * [n_mat, cols / 64, rows].  One kernel; weight preparation, not the hot path.
 * MOE_ERR_BAD_DIMS when cols is not a multiple of 64. */
MOE_API moe_status moe_quantize_nf4(const uint16_t* W, int64_t n_mat, int64_t rows, int32_t cols,
                                    uint8_t* Wq, float* absmax, void* stream);

/* The 16 NF4 code values T[0..15] (host memory, ascending): quantiles of the standard
 * normal distribution at probabilities evenly spaced from delta = 1 - (1/32 + 1/30) / 2
 * towards 1/2 (8 positive values; 7 negative ones, mirrored), an exact zero (T[7]), divided
 * by the largest and rounded to float32, so T[0] = -1 and T[15] = 1.  Host only. */
MOE_API moe_status moe_nf4_codebook(float* values);

/* moe_lora_fwd / moe_lora_bwd with NF4 base weights: Wq_gu [E, H, I] bytes (2I codes per row)
 * and Wq_d [E, I, H / 2] with block scales absmax_gu [E, 2I / 64, H] and absmax_d
 * [E, H / 64, I] (moe_quantize_nf4).  The GEMMs stream the codes (a quarter of the bytes of
 * bf16) and dequantise them to bf16 in shared memory before the tensor cores read them, so
 * the results are bit-identical to moe_lora_fwd / moe_lora_bwd called with the dequantised
 * bf16 weights.  LoRA factors and activations stay bf16; same saved / workspace sizes; SM
 * pairs as for the FP8 forms (MOE_ERR_CUDA where no 2-CTA cluster fits). */
MOE_API moe_status moe_lora_fwd_nf4(const moe_dims* d, const moe_routing* rt, const uint16_t* x,
                                    const uint8_t* Wq_gu, const float* absmax_gu,
                                    const uint16_t* A_gu, const uint16_t* B_gu,
                                    const uint8_t* Wq_d, const float* absmax_d,
                                    const uint16_t* A_d, const uint16_t* B_d, uint16_t* y,
                                    void* saved, size_t saved_bytes,
                                    void* workspace, size_t workspace_bytes,
                                    int32_t* dev_status, void* stream);
MOE_API moe_status moe_lora_bwd_nf4(const moe_dims* d, const moe_routing* rt, const uint16_t* dy,
                                    const uint8_t* Wq_gu, const float* absmax_gu,
                                    const uint16_t* A_gu, const uint16_t* B_gu,
                                    const uint8_t* Wq_d, const float* absmax_d,
                                    const uint16_t* A_d, const uint16_t* B_d,
                                    const void* saved, size_t saved_bytes,
                                    uint16_t* dx, uint16_t* dA_gu, uint16_t* dB_gu,
                                    uint16_t* dA_d, uint16_t* dB_d, float* d_topk_w,
                                    void* workspace, size_t workspace_bytes,
                                    int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------- router
 * The step in front of moe_route: the workloads route each token by a softmax
 * over its E router logits followed by the k largest probabilities.
 *  logits   [T, E] float32 (device)
 *  topk_idx [T, k] int32 out: experts in descending probability; equal logits go
 *           to the lower expert index.  Softmax is strictly increasing in each
 *           logit, so the selection is made on the logits (exact comparisons).
 *  topk_w   [T, k] float32 out: the selected softmax probabilities (fp32), not
 *           renormalised.
 * One kernel, no workspace.  1 <= k <= E <= 1024. */
MOE_API moe_status moe_router_topk(const float* logits, int64_t T, int32_t E, int32_t k,
                                   int32_t* topk_idx, float* topk_w, void* stream);

/* Backward of moe_router_topk with the selection held fixed (the softmax VJP):
 *   d_logits[t,e] = p_e * (g_e - sum_j d_topk_w[t,j] * p_{topk_idx[t,j]}),
 * p = softmax(logits[t]) recomputed in fp32, g_e = d_topk_w[t,j] where
 * topk_idx[t,j] = e (0 elsewhere).  d_logits [T, E] float32 out. */
MOE_API moe_status moe_router_bwd(const float* logits, const int32_t* topk_idx, const float* d_topk_w,
                                  int64_t T, int32_t E, int32_t k, float* d_logits, void* stream);

/* ---------------------------------------------------------------- packed-sequence metadata
 * The "Unsloth and NVIDIA" blog post (section "core idea / structure / how it
 * works", packed-sequence metadata caching): a packed batch concatenates several
 * samples into one token stream, and every layer needs the samples' boundaries
 * (cu_seqlens), the longest sample and the attention structure.  These are the
 * same for all layers of one batch, so they are built once per batch and reused;
 * here on the device, without copies to the host or synchronisation.  The pages
 * do not say how a packed batch is described: read as position ids that restart
 * at 0 at each sample, so a sample starts at token 0 and at every token whose
 * position id is 0.
 *  position_ids [T] int32 or int64 (pos_bytes 4 or 8), device, aligned to its width
 *  cu_seqlens   [T+1] int32 out: entries 0..n are the samples' first tokens, then T
 *               (entries past n are left untouched)
 *  seq_id       [T] int32 out: the sample of each token
 *  n_seqs       [1] int32 out: the number of samples n (0 when T = 0)
 *  max_seqlen   [1] int32 out: the longest sample (0 when T = 0)
 * The outputs are int32 and 4-byte aligned; 0 <= T <= 2^30 (MOE_ERR_BAD_DIMS
 * otherwise).  The caller owns every buffer; one single-CTA kernel, no workspace,
 * enqueued on `stream`. */
MOE_API moe_status moe_packed_metadata(const void* position_ids, int32_t pos_bytes, int64_t T,
                                       int32_t* cu_seqlens, int32_t* seq_id, int32_t* n_seqs,
                                       int32_t* max_seqlen, void* stream);

/* The attention structure of the packed batch, as the dense block-diagonal causal
 * mask that masked attention takes: mask[i * T + j] = 1 when tokens i and j lie in
 * the same sample and j <= i, else 0 (uint8, row-major [T, T]; a torch.bool view).
 * cu_seqlens and seq_id are moe_packed_metadata's outputs for the same batch.
 * mask must be 16-byte aligned and hold T * T bytes; 0 <= T <= 2^30. */
MOE_API moe_status moe_packed_causal_mask(const int32_t* cu_seqlens, const int32_t* seq_id, int64_t T,
                                          uint8_t* mask, void* stream);

/* ---------------------------------------------------------------- diagnostics
 * Per-kernel timing.  moe_timing_enable(1) clears the record and makes every
 * later kernel launch of moe_route / moe_lora_fwd / moe_lora_bwd bracketed by
 * two CUDA events recorded on the caller's stream (the events are created on
 * first use and reused; no device memory is allocated).  moe_timing_enable(0)
 * stops recording.  moe_timing_read(i, ...) reports, for the i-th distinct
 * kernel name recorded, the summed elapsed milliseconds and the number of
 * launches; it WAITS for those events (host-blocking, diagnostics only) and
 * returns MOE_ERR_BAD_DIMS once i is past the last name. */
MOE_API moe_status moe_timing_enable(int32_t on);
MOE_API moe_status moe_timing_read(int32_t index, char* name, size_t name_len,
                                   double* total_ms, int32_t* launches);

/* Number of launch operations (kernels, plus the route's 4-byte memset) the
 * library has issued since it was loaded, counted on the host. */
MOE_API uint64_t moe_launch_count(void);

/* Failure-path test hook.  Every mbarrier wait inside the tensor-core kernels is
 * bounded (2 s); a wait that runs out sets MOE_DEV_TIMEOUT in *dev_status, the
 * kernel stops issuing work, waits (again bounded by 2 s) until the copies and
 * MMAs it already issued have landed, frees its TMEM and returns, so the context
 * stays usable.  This call makes that happen on purpose: the launch_index-th
 * (0-based) launch from now of a single-CTA tensor-core kernel -- a grouped GEMM
 * on single-CTA tiles, a rank-r projection or a LoRA reduction; SM-pair launches
 * are not counted -- bounds its ordinary waits by limit_ns and has its epilogue
 * warps first wait on an mbarrier that nothing arrives on, so those waits run
 * out.  The outputs of the call that contains that launch are unspecified; the
 * next calls are unaffected.  limit_ns in [1000, 2e9] (MOE_ERR_BAD_DIMS
 * otherwise); launch_index < 0 disarms.  Counted on the host, process-wide. */
MOE_API moe_status moe_diag_force_timeout(int32_t launch_index, uint64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LORA_H */
