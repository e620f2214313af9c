// Per-expert LoRA weight gradients on the tensor cores (tcgen05 + TMEM + TMA).
//
//   D[e, j, m] = sum_{p in rows of expert e} Small[p, j] * Big[p, m]
//
// Small = the rank-r activations (already scaled by s), [N, RP]; Big = an
// activation or gradient in sorted row order, [N, M].  The contraction runs
// over the expert's ragged row range, so K differs per expert (0 for an expert
// without rows).  Both operands are MN-major (their contiguous dimension is an
// output dimension): A tile = Big[64 rows, 128 m] as two 64-column boxes with
// 128-byte swizzle, B tile = Small[64 rows, RP].  Rows past the expert's end
// (the next expert's rows, already in the tile) are zeroed in shared memory by
// the MMA warp before the tile is used, so no foreign row enters the sum.
//
// One output tile = (expert, 128 columns of M); each is computed by exactly one
// CTA in a fixed row order: deterministic, no atomics, no split-K.  Experts
// without rows write exact zeros.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>

namespace moe {

namespace {

constexpr int WM = 128, WK = 64;
// Two CTAs per SM: while one is between tiles or waiting for its first loads, the other
// keeps the SM's loads in flight (measured against one CTA per SM: the GPT-OSS-20B-shaped
// reductions 4-5 % faster, the skewed GPT-OSS-120B-shaped ones 11-23 %, the DeepSeek-V3-
// shaped ones 35 %).  A CTA's ring is sized so that two fit in shared memory: 6 stages for
// RP = 16, 5 for 32, 4 for 64.
template <int RP>
__host__ __device__ constexpr int wg_stage_bytes() { return WM * WK * 2 + ((WK * RP * 2 + 1023) / 1024) * 1024; }
template <int RP>
__host__ __device__ constexpr int wg_stages() { return (110 * 1024) / wg_stage_bytes<RP>() < 6 ? (110 * 1024) / wg_stage_bytes<RP>() : 6; }
constexpr int kWThreads = 192;
constexpr int kWABytes = WM * WK * 2;   // 16 KB

// Up to two problems with the same expert partition and rank share one launch.
struct WgradParams {
    CUtensorMap tm_big[2], tm_small[2];
    const int32_t* offsets;
    bf16* D[2];
    int M[2];
    int m_tiles[2];
    int nprob;
    int E, r, rp;
    uint32_t b_sbo, b_swz;
    int32_t* dev_status;
    int64_t N;           // sorted rows (the debug build checks the offsets against it)
    uint64_t wait_ns;    // limit of the ordinary bounded waits
    int stall;           // diagnostics: the epilogue first waits on a barrier nothing arrives on
};

// tile t -> (problem, expert, 128-column tile)
__device__ __forceinline__ void wg_decode(const WgradParams& P, int t, int& prob, int& e, int& mt) {
    const int t0 = P.E * P.m_tiles[0];
    prob = t < t0 ? 0 : 1;
    const int u = prob == 0 ? t : t - t0;
    e = u / P.m_tiles[prob];
    mt = u - e * P.m_tiles[prob];
}

template <int RP>
__global__ void __launch_bounds__(kWThreads, 2) lora_wgrad_tc_kernel(const __grid_constant__ WgradParams P) {
    pdl_wait();      // no early trigger: dependents launch when this long kernel completes
    constexpr int kBBytes = WK * RP * 2;
    constexpr int kStageBytes = wg_stage_bytes<RP>();
    constexpr int kWStages = wg_stages<RP>();
    constexpr int kAcc = RP;
    constexpr uint32_t kTmemCols = (2 * RP < 32) ? 32 : 2 * RP;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kWStages * kStageBytes);
    uint64_t* empty_bar = full_bar + kWStages;
    uint64_t* tfull_bar = empty_bar + kWStages;
    uint64_t* tempty_bar = tfull_bar + 2;
    uint64_t* drain_bar = tempty_bar + 2;            // after an abort: the MMA issuer's last commit
    uint64_t* stall_bar = drain_bar + 1;             // diagnostics: nothing ever arrives on it
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stall_bar + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int32_t* s_off = reinterpret_cast<int32_t*>(tmem_slot + 4);
    static_assert((2 * kWStages + 6) * 8 + 16 <= 256, "barriers and flags fit the 256-byte tail");
    const int E = P.E;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = P.offsets[i];
    if (threadIdx.x == 0) {
        for (int s = 0; s < kWStages; ++s) {
            tc::mbar_init(tc::smem_u32(&full_bar[s]), 1);
            tc::mbar_init(tc::smem_u32(&empty_bar[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(tc::smem_u32(&tfull_bar[a]), 1);
            tc::mbar_init(tc::smem_u32(&tempty_bar[a]), 4);
        }
        tc::mbar_init(tc::smem_u32(drain_bar), 1);
        tc::mbar_init(tc::smem_u32(stall_bar), 1);
        *s_abort = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < P.nprob; ++i) {
            tc::prefetch_tmap(&P.tm_big[i]);
            tc::prefetch_tmap(&P.tm_small[i]);
        }
    }
    if (warp == 1) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    volatile int* s_bad = reinterpret_cast<volatile int*>(tmem_slot + 2);
    if constexpr (MOE_DEBUG) {
        // debug build: offsets that do not describe the N rows schedule no tile
        if (threadIdx.x == 0) *s_bad = dbg_offsets_ok(s_off, nullptr, E, P.N, 1, P.dev_status) ? 0 : 1;
        __syncthreads();
    }
    const int total = (MOE_DEBUG && *s_bad) ? 0 : E * (P.m_tiles[0] + (P.nprob > 1 ? P.m_tiles[1] : 0));
    const uint64_t lim = P.wait_ns;
    int fills = 0;                                   // the producer's stage fills (lane 0 of warp 0)

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int t = blockIdx.x; t < total && !*s_abort; t += gridDim.x) {
                int prob, e, mt;
                wg_decode(P, t, prob, e, mt);
                const int beg = s_off[e], end = s_off[e + 1];
                for (int p0 = beg; p0 < end; p0 += WK) {
                    if (!tc::mbar_wait(tc::smem_u32(&empty_bar[stage]), phase ^ 1, lim)) {
                        *s_abort = 1;
                        atomicOr(P.dev_status, MOE_DEV_TIMEOUT);
                        break;
                    }
                    const uint32_t fb = tc::smem_u32(&full_bar[stage]);
                    const uint32_t sa = tc::smem_u32(smem + stage * kStageBytes);
                    tc::mbar_arrive_expect_tx(fb, kWABytes + kBBytes);
                    tc::tma_load_2d(sa, &P.tm_big[prob], fb, mt * WM, p0);
                    tc::tma_load_2d(sa + kWABytes / 2, &P.tm_big[prob], fb, mt * WM + 64, p0);
                    tc::tma_load_2d(sa + kWABytes, &P.tm_small[prob], fb, 0, p0);
                    ++fills;
                    if (++stage == kWStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        }
    } else if (warp == 1) {
        const uint32_t idesc = tc::idesc_bf16(WM, RP, true, true);
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        for (int t = blockIdx.x; t < total && !*s_abort; t += gridDim.x) {
            int prob, e, mt;
            wg_decode(P, t, prob, e, mt);
            const int beg = s_off[e], end = s_off[e + 1];
            if (end == beg) continue;                       // written as zeros by the epilogue
            const int acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            ++it;
            bool ok = tc::mbar_wait(tc::smem_u32(&tempty_bar[acc]), acc_phase ^ 1, lim);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) {
                    *s_abort = 1;
                    atomicOr(P.dev_status, MOE_DEV_TIMEOUT);
                }
                break;
            }
            tc::fence_after_sync();
            const uint32_t d = tmem_base + acc * kAcc;
            for (int p0 = beg; p0 < end; p0 += WK) {
                ok = tc::mbar_wait(tc::smem_u32(&full_bar[stage]), phase, lim);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    if (lane == 0) {
                        *s_abort = 1;
                        atomicOr(P.dev_status, MOE_DEV_TIMEOUT);
                    }
                    break;
                }
                const uint32_t sa = tc::smem_u32(smem + stage * kStageBytes);
                const uint32_t sb = sa + kWABytes;
                const int valid = min(WK, end - p0);
                if (valid < WK) {
                    // zero the rows of B that belong to the next expert (whole rows: the
                    // swizzle only permutes 16-byte chunks inside a row)
                    uint8_t* bt = smem + stage * kStageBytes + kWABytes;
                    const int nbytes = (WK - valid) * RP * 2;
                    for (int i = lane * 16; i < nbytes; i += 32 * 16)
                        *reinterpret_cast<uint4*>(bt + valid * RP * 2 + i) = make_uint4(0, 0, 0, 0);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                __syncwarp();
                tc::fence_after_sync();
                if (lane == 0) {
#pragma unroll
                    for (int kk = 0; kk < WK / 16; ++kk) {
                        const uint64_t ad = tc::smem_desc(sa + kk * 2048, kWABytes / 2, 1024, tc::kSw128);
                        const uint64_t bd = tc::smem_desc(sb + kk * 16 * RP * 2, kBBytes, P.b_sbo, P.b_swz);
                        tc::mma_bf16(d, ad, bd, idesc, (p0 > beg || kk > 0) ? 1u : 0u);
                    }
                    tc::mma_commit(tc::smem_u32(&empty_bar[stage]));
                }
                __syncwarp();
                if (++stage == kWStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
            if (lane == 0) tc::mma_commit(tc::smem_u32(&tfull_bar[acc]));
            __syncwarp();
        }
    } else {
        const int q = warp & 3;
        const int row = q * 32 + lane;
        int it = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            int prob, e, mt;
            wg_decode(P, t, prob, e, mt);
            const int M = P.M[prob];
            const int m = mt * WM + row;
            bf16* De = P.D[prob] + (int64_t)e * P.r * M;
            if (s_off[e + 1] == s_off[e]) {
                if (m < M)
                    for (int j = 0; j < P.r; ++j) De[(int64_t)j * M + m] = f2bf(0.f);
                continue;
            }
            const int acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            ++it;
            // diagnostics: a launch chosen to fail first waits on a barrier nothing arrives on
            const bool ok = (P.stall == 0 || tc::mbar_wait(tc::smem_u32(stall_bar), 0, lim)) &&
                            tc::mbar_wait(tc::smem_u32(&tfull_bar[acc]), acc_phase, lim);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) {
                    *s_abort = 1;
                    atomicOr(P.dev_status, MOE_DEV_TIMEOUT);
                }
                break;
            }
            tc::fence_after_sync();
            const uint32_t tb = tmem_base + acc * kAcc + ((uint32_t)(q * 32) << 16);
#pragma unroll
            for (int c = 0; c < RP; c += 16) {
                float v[16];
                tc::tmem_ld16(tb + c, v);
                tc::tmem_ld_wait();
                if (m < M) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (c + i < P.r) De[(int64_t)(c + i) * M + m] = f2bf(v[i]);
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(tc::smem_u32(&tempty_bar[acc]));
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    // ---- abort drain: the loads of the last stages may be unconsumed and the last MMAs
    // unread; every one has landed before the shared memory and TMEM are released (full limit)
    if (*s_abort) {
        if (warp == 0 && lane == 0) {
            // every fill before fills - kWStages was consumed by the MMA warp; the later ones
            // are the current phases of their stages, each completed by its loads alone
            for (int f = max(0, fills - kWStages); f < fills; ++f)
                tc::mbar_wait(tc::smem_u32(&full_bar[f % kWStages]), (uint32_t)(f / kWStages) & 1u);
        } else if (warp == 1 && lane == 0) {
            tc::mma_commit(tc::smem_u32(drain_bar));
            tc::mbar_wait(tc::smem_u32(drain_bar), 0);
        }
        tc::fence_before_sync();
        __syncthreads();
    }
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem_base, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 wg_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool encode2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_in, uint32_t box_out,
              CUtensorMapSwizzle sw) {
    auto fn = wg_encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t gd[2] = {inner, outer};
    cuuint64_t gs[1] = {inner * 2};
    cuuint32_t bx[2] = {box_in, box_out};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gd, gs, bx, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int wg_sm_count() {
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

template <int RP>
cudaError_t launch_wg(const WgradParams& P, cudaStream_t s) {
    const size_t smem = 1024 + (size_t)wg_stages<RP>() * wg_stage_bytes<RP>() + 256 + (size_t)(P.E + 1) * sizeof(int32_t);
    auto k = lora_wgrad_tc_kernel<RP>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // all of the SM's unified memory as shared memory, so that two CTAs fit
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    // Two CTAs per SM.  The runtime's occupancy query reports one for this kernel at any
    // shared-memory size, but the grid of two per SM measured faster on every workload (see
    // above); no CTA waits on another, so the launch is correct however many are resident.
    const int total = P.E * (P.m_tiles[0] + (P.nprob > 1 ? P.m_tiles[1] : 0));
    const int grid = std::min(2 * wg_sm_count(), total);
    return launch_pdl(k, dim3(grid), dim3(kWThreads), smem, s, P);
}

}  // namespace

cudaError_t launch_lora_wgrad_tc(const WgradProblem* probs, int nprob, int rp, int r, const int32_t* offsets, int E,
                                 int64_t N, int32_t* dev_status, cudaStream_t s) {
    if (nprob < 1 || nprob > 2 || (rp != 16 && rp != 32 && rp != 64)) return cudaErrorInvalidValue;
    WgradParams P;
    memset(&P, 0, sizeof(P));
    P.offsets = offsets;
    P.nprob = nprob;
    P.E = E; P.r = r; P.rp = rp;
    P.dev_status = dev_status;
    P.N = N;
    P.wait_ns = tc::kWaitTimeoutNs;
    P.b_sbo = 8 * rp * 2;
    P.b_swz = rp >= 64 ? tc::kSw128 : (rp >= 32 ? tc::kSw64 : tc::kSw32);
    const CUtensorMapSwizzle bsw = rp >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                            : (rp >= 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
    const uint64_t rows = N > 0 ? (uint64_t)N : 1;
    for (int i = 0; i < nprob; ++i) {
        const WgradProblem& q = probs[i];
        if (q.M % 64 != 0) return cudaErrorInvalidValue;
        P.D[i] = (bf16*)q.D;
        P.M[i] = q.M;
        P.m_tiles[i] = (q.M + WM - 1) / WM;
        if (!encode2d(&P.tm_big[i], q.Big, (uint64_t)q.M, rows, 64, WK, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        if (!encode2d(&P.tm_small[i], q.Small, (uint64_t)rp, rows, (uint32_t)rp, WK, bsw)) return cudaErrorInvalidValue;
    }
    // diagnostics: a launch the caller chose to fail (moe_diag_force_timeout)
    const DiagWait dw = diag_next_single_cta_launch();
    if (dw.stall) {
        P.stall = 1;
        P.wait_ns = dw.limit_ns;
    }
    switch (rp) {
        case 16: return launch_wg<16>(P, s);
        case 32: return launch_wg<32>(P, s);
        default: return launch_wg<64>(P, s);
    }
}

}  // namespace moe
