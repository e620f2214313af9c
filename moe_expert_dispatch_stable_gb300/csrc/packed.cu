// Packed-sequence metadata, built once per packed batch on the device.
//
// The "Unsloth and NVIDIA" blog post (section "core idea / structure / how it
// works", packed-sequence metadata caching): a packed batch concatenates several
// samples into one token stream, and every layer needs the samples' boundaries
// (cu_seqlens), the longest sample and the attention structure.  They are the
// same for all layers of one batch, so they are built once and reused, instead of
// being prepared again in every layer with device-to-host copies.  Here both steps
// stay on the device and never synchronise with the host:
//
//   packed_meta   one CTA walks the tokens in chunks of 4096: a token starts a
//                 sample when it is token 0 or its position id is 0; a block-wide
//                 exclusive scan of those flags (carried across chunks) gives each
//                 token's sample id and each sample's first token; then the CTA
//                 reduces the sample lengths to the longest one.
//   packed_mask   the block-diagonal causal mask, 16 bytes per thread: row i holds
//                 ones exactly in the columns [cu_seqlens[seq_id[i]], i] (row by row
//                 when T is a multiple of 16, else over the flat byte array).
#include "common.cuh"
#include "kernels.h"

#include <algorithm>

namespace moe {

namespace {

constexpr int kMetaThreads = 1024;
constexpr int kMetaItems = 4;                              // tokens per thread and chunk
constexpr int kMetaChunk = kMetaThreads * kMetaItems;
constexpr int kMaskThreads = 256;

// Block-wide exclusive scan of one int per thread; *total gets the block's sum.
// Every thread of the block must call it; it ends with a barrier.
__device__ int meta_exclusive_scan(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += n;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = (blockDim.x + 31) >> 5;
        const int s = lane < nw ? warp_sums[lane] : 0;
        int si = s;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, si, d);
            if (lane >= d) si += n;
        }
        if (lane < nw) warp_sums[lane] = si - s;
        if (lane == nw - 1) *total = si;
    }
    __syncthreads();
    const int out = warp_sums[warp] + incl - v;
    __syncthreads();
    return out;
}

template <typename PosT>
__global__ void __launch_bounds__(kMetaThreads)
packed_meta_kernel(const PosT* __restrict__ pos, int T, int32_t* __restrict__ cu_seqlens,
                   int32_t* __restrict__ seq_id, int32_t* __restrict__ n_seqs, int32_t* __restrict__ max_seqlen) {
    pdl_wait();
    pdl_trigger();
    __shared__ int warp_sums[32];
    __shared__ int total;
    __shared__ int warp_max[32];
    int carry = 0;                                         // samples started before this chunk
    for (int base = 0; base < T; base += kMetaChunk) {     // uniform trip count
        const int t0 = base + (int)threadIdx.x * kMetaItems;
        int flag[kMetaItems];
        int c = 0;
#pragma unroll
        for (int j = 0; j < kMetaItems; ++j) {
            const int t = t0 + j;
            flag[j] = t < T && (t == 0 || pos[t] == 0) ? 1 : 0;
            c += flag[j];
        }
        int run = carry + meta_exclusive_scan(c, warp_sums, &total);
#pragma unroll
        for (int j = 0; j < kMetaItems; ++j) {
            const int t = t0 + j;
            if (t < T) {
                run += flag[j];
                seq_id[t] = run - 1;
                if (flag[j]) cu_seqlens[run - 1] = t;
            }
        }
        carry += total;
    }
    const int n = carry;
    if (threadIdx.x == 0) {
        cu_seqlens[n] = T;
        *n_seqs = n;
    }
    __syncthreads();                                       // every cu_seqlens entry is visible to the block
    int mx = 0;
    for (int s = threadIdx.x; s < n; s += blockDim.x) mx = max(mx, cu_seqlens[s + 1] - cu_seqlens[s]);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, d));
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x < 32) {
        mx = threadIdx.x < (blockDim.x >> 5) ? warp_max[threadIdx.x] : 0;
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, d));
        if (threadIdx.x == 0) *max_seqlen = mx;
    }
}

// mask[f] for the flat byte f = i * T + j: 1 iff cu_seqlens[seq_id[i]] <= j <= i.
__global__ void __launch_bounds__(kMaskThreads)
packed_mask_kernel(const int32_t* __restrict__ cu_seqlens, const int32_t* __restrict__ seq_id, int64_t T,
                   uint8_t* __restrict__ mask) {
    pdl_wait();
    pdl_trigger();
    const int64_t nbytes = T * T;
    const int64_t nchunks = (nbytes + 15) / 16;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < nchunks; q += stride) {
        const int64_t f0 = q * 16;
        int64_t i = f0 / T;
        int64_t j = f0 - i * T;
        // debug build: a sample id outside [0, T] gives the row no ones
        int64_t lo = dbg_index_ok(seq_id[i], T + 1, nullptr) ? cu_seqlens[seq_id[i]] : i + 1;
        uint32_t w[4] = {0u, 0u, 0u, 0u};                  // byte u of the chunk in w[u / 4]
        const int nb = (int)min((int64_t)16, nbytes - f0);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            if (u < nb && j >= lo && j <= i) w[u >> 2] |= 1u << ((u & 3) * 8);
            if (++j == T && u + 1 < nb) {
                j = 0;
                ++i;
                lo = dbg_index_ok(seq_id[i], T + 1, nullptr) ? cu_seqlens[seq_id[i]] : i + 1;
            }
        }
        if (nb == 16) {
            *reinterpret_cast<uint4*>(mask + f0) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
#pragma unroll
            for (int u = 0; u < 16; ++u)
                if (u < nb) mask[f0 + u] = (uint8_t)((w[u >> 2] >> ((u & 3) * 8)) & 1u);
        }
    }
}

// T % 16 == 0: every 16-byte chunk lies inside one row.  Rows are spread over the grid;
// within a row, lo = cu_seqlens[seq_id[i]] is looked up once and each chunk is all zeros,
// all ones, or (at most two chunks per row) mixed.
__global__ void __launch_bounds__(kMaskThreads)
packed_mask_rows_kernel(const int32_t* __restrict__ cu_seqlens, const int32_t* __restrict__ seq_id, int T,
                        uint8_t* __restrict__ mask) {
    pdl_wait();
    pdl_trigger();
    const int chunks = T >> 4;
    for (int i = blockIdx.x; i < T; i += gridDim.x) {
        const int lo = dbg_index_ok(seq_id[i], (int64_t)T + 1, nullptr) ? cu_seqlens[seq_id[i]] : i + 1;
        uint4* row = reinterpret_cast<uint4*>(mask + (int64_t)i * T);
        for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
            const int j0 = c << 4;
            uint4 v;
            if (j0 + 15 < lo || j0 > i) {
                v = make_uint4(0u, 0u, 0u, 0u);
            } else if (j0 >= lo && j0 + 15 <= i) {
                v = make_uint4(0x01010101u, 0x01010101u, 0x01010101u, 0x01010101u);
            } else {
                uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    if (j0 + u >= lo && j0 + u <= i) w[u >> 2] |= 1u << ((u & 3) * 8);
                v = make_uint4(w[0], w[1], w[2], w[3]);
            }
            row[c] = v;
        }
    }
}

int mask_sm_count() {
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

}  // namespace

cudaError_t launch_packed_metadata(const void* position_ids, int pos_bytes, int64_t T, int32_t* cu_seqlens,
                                   int32_t* seq_id, int32_t* n_seqs, int32_t* max_seqlen, cudaStream_t s) {
    if (pos_bytes == 8)
        return launch_pdl(packed_meta_kernel<long long>, dim3(1), dim3(kMetaThreads), 0, s,
                          (const long long*)position_ids, (int)T, cu_seqlens, seq_id, n_seqs, max_seqlen);
    return launch_pdl(packed_meta_kernel<int32_t>, dim3(1), dim3(kMetaThreads), 0, s, (const int32_t*)position_ids,
                      (int)T, cu_seqlens, seq_id, n_seqs, max_seqlen);
}

cudaError_t launch_packed_mask(const int32_t* cu_seqlens, const int32_t* seq_id, int64_t T, uint8_t* mask,
                               cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (T % 16 == 0) {
        const int64_t blocks = std::min<int64_t>(T, (int64_t)mask_sm_count() * 16);
        return launch_pdl(packed_mask_rows_kernel, dim3((unsigned)blocks), dim3(kMaskThreads), 0, s, cu_seqlens,
                          seq_id, (int)T, mask);
    }
    const int64_t nchunks = (T * T + 15) / 16;
    const int64_t blocks = std::min<int64_t>((nchunks + kMaskThreads - 1) / kMaskThreads, (int64_t)mask_sm_count() * 8);
    return launch_pdl(packed_mask_kernel, dim3((unsigned)blocks), dim3(kMaskThreads), 0, s, cu_seqlens, seq_id, T,
                      mask);
}

}  // namespace moe
