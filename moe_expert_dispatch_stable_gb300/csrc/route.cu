// Routing: group the T*k routed slots by expert, on the device, with no host sync.
//
// The Unsloth x NVIDIA blog post (section "core idea / structure / how it
// works", GPT-OSS MoE routing paragraphs) replaces one torch.where query per
// expert by: flatten the top-k assignment, stable-sort it by expert id,
// bincount once, slice by offsets.  Here the three steps are two kernels:
//
//   route_count   each CTA histograms a 1024-slot chunk (warp-aggregated with
//                 __match_any_sync into shared-memory counters) and writes its
//                 per-expert counts; the last CTA to finish (atomic ticket after
//                 a fence; no spinning) sums them, scans them to offsets and
//                 tile offsets and turns the per-CTA counts into each CTA's
//                 starting position relative to every expert segment (the
//                 scatter adds the segment's offset).
//   route_scatter each CTA re-reads its chunk; every warp owns a contiguous
//                 64-slot sub-chunk, so a slot's position is
//                   CTA base[e] + earlier warps' count[e] + earlier rounds' count[e]
//                   + lanes below it with the same expert (popc of the match mask)
//                 which is exactly its rank among equal keys in flat order: a
//                 stable counting sort.
#include "common.cuh"
#include "kernels.h"

#include <cuda.h>
#include <mutex>

namespace moe {

constexpr int kRouteChunk = 1024;            // slots per CTA: >= 16 CTAs at 16K slots
constexpr int kCountThreads = 1024;
constexpr int kScatterThreads = 512;                  // 16 warps x 64 slots
constexpr int kScatterWarps = kScatterThreads / 32;
constexpr int kSlotsPerWarp = kRouteChunk / kScatterWarps;

template <typename IdxT>
__device__ __forceinline__ int load_expert(const IdxT* idx, int64_t i, int64_t end, int E, bool& bad) {
    if (i >= end) return -1;
    long long v = (long long)idx[i];
    if (v < 0 || v >= E) { bad = true; return -1; }
    return (int)v;
}

// Block-wide exclusive scan of one int per thread (blockDim.x <= 1024).
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += n;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = (blockDim.x + 31) >> 5;
        int s = lane < nw ? warp_sums[lane] : 0;
        int si = s;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, si, d);
            if (lane >= d) si += n;
        }
        if (lane < nw) warp_sums[lane] = si - s;      // exclusive warp offsets
        if (lane == nw - 1) *total = si;
    }
    __syncthreads();
    int out = warp_sums[warp] + incl - v;
    __syncthreads();
    return out;
}

template <typename IdxT>
__global__ void __launch_bounds__(kCountThreads)
route_count_kernel(const IdxT* __restrict__ idx, int64_t N, int E,
                   int32_t* __restrict__ block_counts, unsigned int* __restrict__ ticket,
                   int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                   int32_t* __restrict__ tile_offsets, int32_t* __restrict__ dev_status) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int32_t hist[];                  // [E]
    __shared__ int warp_sums[32];
    __shared__ int scan_total;
    __shared__ bool is_last;
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();

    const int64_t beg = (int64_t)blockIdx.x * kRouteChunk;
    const int64_t end = min(N, beg + kRouteChunk);
    bool bad = false;
    for (int64_t base = beg; base < end; base += blockDim.x) {   // uniform trip count
        const int e = load_expert(idx, base + threadIdx.x, end, E, bad);
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[e], __popc(peers));
    }
    if (bad) atomicOr(dev_status, MOE_DEV_BAD_EXPERT_ID);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) block_counts[(int64_t)blockIdx.x * E + e] = hist[e];

    // last CTA to arrive does the scan (threadFenceReduction pattern, no waiting)
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = (atomicAdd(ticket, 1u) == gridDim.x - 1);
    __syncthreads();
    if (!is_last) return;
    __threadfence();

    const int nb = gridDim.x;
    const int e = threadIdx.x;                         // E <= blockDim.x
    int run = 0;
    if (e < E) {
        // exclusive prefix over the CTAs within expert e; each batch issues all its loads
        // before its stores, so a batch costs one L2 round trip instead of one per CTA
        constexpr int kBatch = 16;
        for (int b0 = 0; b0 < nb; b0 += kBatch) {
            const int nbat = min(kBatch, nb - b0);
            int c[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) c[j] = j < nbat ? __ldcg(block_counts + (int64_t)(b0 + j) * E + e) : 0;
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                if (j < nbat) block_counts[(int64_t)(b0 + j) * E + e] = run;
                run += c[j];
            }
        }
    }
    const int off = block_exclusive_scan(e < E ? run : 0, warp_sums, &scan_total);
    const int tiles = e < E ? (run + kTileM - 1) / kTileM : 0;
    const int toff = block_exclusive_scan(tiles, warp_sums, &scan_total);
    if (e < E) {
        counts[e] = run;
        offsets[e] = off;                              // the scatter adds it to each CTA's base
        tile_offsets[e] = toff;
    }
    if (e == E - 1) {
        offsets[E] = off + run;
        tile_offsets[E] = toff + tiles;
    }
    if (threadIdx.x == 0) *ticket = 0u;                // leave the ticket ready for the next call
}

template <typename IdxT>
__global__ void __launch_bounds__(kScatterThreads)
route_scatter_kernel(const IdxT* __restrict__ idx, const float* __restrict__ topk_w, int64_t N, int E,
                     const int32_t* __restrict__ block_base, const int32_t* __restrict__ offsets,
                     int32_t* __restrict__ perm, int32_t* __restrict__ inv_perm,
                     float* __restrict__ w_sorted) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int32_t wcnt[];                  // [kScatterWarps][E]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kScatterWarps * E; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();

    const int64_t beg = (int64_t)blockIdx.x * kRouteChunk;
    const int64_t end = min(N, beg + kRouteChunk);
    const int64_t wbeg = beg + (int64_t)warp * kSlotsPerWarp;
    int32_t* my = wcnt + warp * E;
    bool bad = false;
    // 1) per-warp histogram of its sub-chunk
    for (int rr = 0; rr < kSlotsPerWarp; rr += 32) {
        const int e = load_expert(idx, wbeg + rr + lane, min(end, wbeg + kSlotsPerWarp), E, bad);
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // 2) exclusive scan over warps, seeded with this CTA's base inside each segment
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = offsets[e] + block_base[(int64_t)blockIdx.x * E + e];
        for (int w = 0; w < kScatterWarps; ++w) {
            const int c = wcnt[w * E + e];
            wcnt[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    // 3) rank = running base + lanes below with the same expert
    const unsigned lt = (1u << lane) - 1u;
    for (int rr = 0; rr < kSlotsPerWarp; rr += 32) {
        const int64_t i = wbeg + rr + lane;
        const int e = load_expert(idx, i, min(end, wbeg + kSlotsPerWarp), E, bad);
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        int pos = 0;
        if (e >= 0) pos = my[e] + __popc(peers & lt);
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
        __syncwarp();
        if (e >= 0) {
            perm[pos] = (int32_t)i;
            inv_perm[i] = pos;
            w_sorted[pos] = topk_w[i];
        }
    }
}

size_t route_workspace_bytes(int64_t N, int E) {
    const int64_t nb = N > 0 ? (N + kRouteChunk - 1) / kRouteChunk : 1;
    return align_up((size_t)nb * E * sizeof(int32_t), 256) + 256;
}

cudaError_t launch_route(const void* idx, int idx_bytes, const float* topk_w, int64_t N, int E,
                         const moe_routing& out, void* ws, int32_t* dev_status, cudaStream_t s) {
    const int nb = N > 0 ? (int)((N + kRouteChunk - 1) / kRouteChunk) : 1;
    int32_t* block_counts = (int32_t*)ws;
    unsigned int* ticket = (unsigned int*)((char*)ws + align_up((size_t)nb * E * sizeof(int32_t), 256));
    cudaError_t err = cudaMemsetAsync(ticket, 0, sizeof(unsigned int), s);
    if (err != cudaSuccess) return err;
    const size_t sm_count = (size_t)E * sizeof(int32_t);
    const size_t sm_scatter = (size_t)kScatterWarps * E * sizeof(int32_t);
    auto run = [&](auto kc, auto ks, const auto* ix) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_scatter);
        if (e != cudaSuccess) return e;
        e = launch_pdl(kc, dim3(nb), dim3(kCountThreads), sm_count, s, ix, N, E, block_counts, ticket, out.counts,
                       out.offsets, out.tile_offsets, dev_status);
        if (e != cudaSuccess || N == 0) return e;
        return launch_pdl(ks, dim3(nb), dim3(kScatterThreads), sm_scatter, s, ix, topk_w, N, E,
                          (const int32_t*)block_counts, (const int32_t*)out.offsets, out.perm, out.inv_perm,
                          out.w_sorted);
    };
    if (idx_bytes == 8)
        return run(route_count_kernel<long long>, route_scatter_kernel<long long>, (const long long*)idx);
    return run(route_count_kernel<int32_t>, route_scatter_kernel<int32_t>, (const int32_t*)idx);
}

// ---------------------------------------------------------------- fixed scratch
// Scratch of moe_route_static: the per-CTA histograms and the ticket live in this
// file-scope device array instead of a caller-provided workspace.  Every GPU that
// loads the library holds it until the process exits; every call shares it.
static __device__ __align__(256) unsigned char g_route_scratch[MOE_ROUTE_STATIC_SCRATCH_BYTES];

// The driver's cuCtxGetCurrent, looked up once through the runtime (no link to libcuda).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

// Device address of g_route_scratch in the current context.  The host-side name of
// the array is only a stand-in, so the address is looked up (with the device current)
// and cached per device together with the context it belongs to; a new context on the
// device (after cudaDeviceReset, or a primary context destroyed and made again) is
// looked up afresh.
cudaError_t route_static_scratch(void** ptr) {
    static std::mutex mu;
    static void* cached[64] = {nullptr};
    static CUcontext cached_ctx[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const CtxGetCurrentFn get = ctx_get_current();
    if (get == nullptr) return cudaErrorInitializationError;
    CUcontext ctx = nullptr;                  // NULL before the runtime made a context current
    if (get(&ctx) != CUDA_SUCCESS) return cudaErrorInitializationError;
    std::lock_guard<std::mutex> g(mu);
    if (ctx == nullptr || cached[dev] == nullptr || cached_ctx[dev] != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_route_scratch);     // makes the primary context current if needed
        if (e != cudaSuccess) return e;
        if (ctx == nullptr && (get(&ctx) != CUDA_SUCCESS || ctx == nullptr)) return cudaErrorInitializationError;
        cached[dev] = p;
        cached_ctx[dev] = ctx;
    }
    *ptr = cached[dev];
    return cudaSuccess;
}

}  // namespace moe
