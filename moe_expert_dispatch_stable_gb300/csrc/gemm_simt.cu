// Grouped GEMM, CUDA-core version: 64x64 output tiles, one expert per tile,
// fp32 accumulation.  Same problem and epilogues as the tcgen05 engine; kept
// as the numerics reference of that engine (selected with
// launch_grouped_gemm_simt) and used by the tests.
#include "common.cuh"
#include "kernels.h"
#include "epilogue.cuh"

namespace moe {

namespace {
constexpr int BM = 64, BN = 64, BK = 16, NT = 256;
}

template <int EPI>
__global__ void __launch_bounds__(NT) grouped_gemm_simt_kernel(const GroupedGemm g) {
    constexpr bool PAIRED = (EPI == EPI_SWIGLU);
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN];
    __shared__ float Bs2[PAIRED ? BK : 1][BN];
    __shared__ int s_e, s_mt;

    // map blockIdx.x -> (expert, 64-row tile of that expert)
    if (threadIdx.x == 0) {
        int t = blockIdx.x, cum = 0, e_found = -1, mt = 0;
        for (int e = 0; e < g.E; ++e) {
            const int n = g.offsets[e + 1] - g.offsets[e];
            const int nt = (n + BM - 1) / BM;
            if (t < cum + nt) { e_found = e; mt = t - cum; break; }
            cum += nt;
        }
        s_e = e_found;
        s_mt = mt;
    }
    __syncthreads();
    const int e = s_e;
    if (e < 0) return;
    const int row0 = g.offsets[e] + s_mt * BM;
    const int row_end = g.offsets[e + 1];
    const int n0 = blockIdx.y * BN;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;

    const bf16* A = (const bf16*)g.A;
    const bf16* B = (const bf16*)g.B + (int64_t)e * g.b_expert_stride;
    float acc[4][4] = {}, acc2[4][4] = {};

    auto run = [&](const bf16* Ap, int lda, int K, const bf16* Bp, bool mn, int ldb) {
        for (int k0 = 0; k0 < K; k0 += BK) {
            for (int i = threadIdx.x; i < BM * BK; i += NT) {
                const int rr = i / BK, kk = i % BK;
                const int p = row0 + rr, c = k0 + kk;
                As[kk][rr] = (p < row_end && c < K) ? bf2f(Ap[(int64_t)p * lda + c]) : 0.f;
            }
            for (int i = threadIdx.x; i < BK * BN; i += NT) {
                const int kk = i / BN, nn = i % BN;
                const int n = n0 + nn, c = k0 + kk;
                float v = 0.f, v2 = 0.f;
                if (n < g.Ncols && c < K) {
                    v = bf2f(mn ? Bp[(int64_t)c * ldb + n] : Bp[(int64_t)n * ldb + c]);
                    if (PAIRED) v2 = bf2f(mn ? Bp[(int64_t)c * ldb + n + g.Ncols] : Bp[(int64_t)(n + g.Ncols) * ldb + c]);
                }
                Bs[kk][nn] = v;
                if (PAIRED) Bs2[kk][nn] = v2;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < BK; ++kk) {
                float a[4], b[4], b2[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    b[j] = Bs[kk][tx * 4 + j];
                    if (PAIRED) b2[j] = Bs2[kk][tx * 4 + j];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
                        if (PAIRED) acc2[i][j] = fmaf(a[i], b2[j], acc2[i][j]);
                    }
            }
            __syncthreads();
        }
    };
    run(A, g.K, g.K, B, g.b_mn_major, g.ldb);
    if (g.A2 != nullptr && g.r > 0)
        run((const bf16*)g.A2, g.rp, g.r, (const bf16*)g.B2 + (int64_t)e * g.b2_expert_stride, true, g.ldb2);

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int p = row0 + ty * 4 + i;
        if (p >= row_end) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= g.Ncols) continue;
            epilogue_store<EPI>(g, p, n, acc[i][j], acc2[i][j]);
        }
    }
}

cudaError_t launch_grouped_gemm_simt(const GroupedGemm& g, cudaStream_t s) {
    if (g.N == 0) return cudaSuccess;
    const int64_t max_tiles = (g.N + BM - 1) / BM + g.E;
    dim3 grid((unsigned)max_tiles, (g.Ncols + BN - 1) / BN);
    switch (g.epi) {
        case EPI_SWIGLU: grouped_gemm_simt_kernel<EPI_SWIGLU><<<grid, NT, 0, s>>>(g); break;
        case EPI_ROWSCALE_F32: grouped_gemm_simt_kernel<EPI_ROWSCALE_F32><<<grid, NT, 0, s>>>(g); break;
        case EPI_DSWIGLU: grouped_gemm_simt_kernel<EPI_DSWIGLU><<<grid, NT, 0, s>>>(g); break;
        default: grouped_gemm_simt_kernel<EPI_F32><<<grid, NT, 0, s>>>(g); break;
    }
    return cudaGetLastError();
}

}  // namespace moe
