// Grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// All experts' weights are one stacked tensor and the group sizes are the
// routing counts (the Unsloth 2026 wiki page, section "Optimisation 3:
// grouped_mm and Split-LoRA for MoE training"): one persistent launch covers
// every (expert, 128-row tile, output-column tile).  The scheduler reads the
// expert offsets and tile offsets that moe_route wrote to device memory, so
// the host never learns the group sizes.  Split-LoRA: the rank-r product is
// one more K step of the same accumulator (A2 = s * x A^T rows, B2 = B), so
// W + BA is never formed.
//
// CTA = 10 warps, one CTA per SM, grid = #SMs:
//   warp 0      TMA producer (one lane): A [128 x 64] and B [256 x 64] per stage,
//               4 stages of 48 KB, 128-byte swizzle; the LoRA step loads A2 / B2
//               (SM pairs: 3 stages of two 32 KB k-blocks, see Geo)
//   warp 1      TMEM allocator + MMA issuer (one lane): 4 x tcgen05.mma
//               M=128 N=256 K=16 per stage into one of two 256-column fp32
//               accumulators (double buffer: the epilogue of tile i overlaps
//               the MMAs of tile i+1)
//   warps 2..9  epilogue (two per TMEM lane quarter, each half the columns):
//               tcgen05.ld 32 lanes x 16 columns, fused SwiGLU / routing-weight
//               scale / SwiGLU backward, masked stores
// Quantised base weights (e4m3 or NF4 codes, SM pairs only): 18 warps, warps 2..5
// the epilogue (one per lane quarter) and warps 6..17 three groups of converters that
// expand each stage's codes into bf16 B tiles in shared memory.
// Every mbarrier wait is bounded; a wait that gives up sets MOE_DEV_TIMEOUT.
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>

namespace moe {

namespace {

constexpr int BM = 128, BK = 64;
// Quantised weights add CG groups of 4 converter warps (CG = 0 with bf16 weights).  A group
// g owns the stages s with s % CG == g, so that several stages are dequantised at once and
// each stage's fixed costs (the wait, two group barriers, the proxy fence, the signal)
// overlap other groups' work; owning whole stages keeps every mbarrier phase wait of a
// group within one phase of the barrier (a stage cannot move on before its owner has
// arrived).  Epilogue warps: 2 per TMEM lane quarter, each half the columns, except with 3
// converter groups: 1 per lane quarter, so that the CTA stays at 576 threads (the register
// budget: 96 registers a thread).  Three groups suit long k loops, whose tiles give the
// slower 4-warp epilogue time to finish (see launch_impl).
__host__ __device__ constexpr int epi_warps(int cg) { return cg == 3 ? 4 : 8; }
__host__ __device__ constexpr int threads_of(int cg) { return 64 + 32 * epi_warps(cg) + 128 * cg; }
constexpr int kSignalBytes = 4;                // quantised pairs: the peer's "B half converted" store
constexpr unsigned kPaceNs = 500;              // epilogue store pacing (see the epilogue)
constexpr int kABytes = BM * BK * 2;         // 16 KB
constexpr int kBoxMN = 64 * BK * 2;          // one 64-column MN-major box of B: 8 KB

// Tile geometry for an output tile width BN (256 for the expert GEMMs; 16/32/64
// for the rank-r projections).  PAIR: a 2-CTA cluster shares one 256 x 256 tile,
// each CTA holding 128 rows of A and 128 columns of B per stage.
template <int BN, bool PAIR = false, int QB = 0>
struct Geo {
    // narrow tiles (the HBM-bound projections) load KW 64-column boxes of A per stage so
    // that every row is fetched in 256-512 byte runs
    static constexpr int KW = BN >= 256 ? 1 : (BN <= 16 ? 4 : 2);
    static constexpr int kBBytes = (PAIR ? BN / 2 : BN) * BK * 2 * KW;
    // quantised weights (QB-bit codes: 8 = e4m3, 4 = NF4): the TMA lands the codes at the
    // top of the B slot and the converter warps expand them in place, so a stage is as
    // large as with bf16 weights
    static constexpr int kQBytes = QB ? kBBytes * QB / 16 : 0;
    // bf16 SM pairs take two 64-deep k-blocks per ring stage: one barrier wait, 8 MMAs
    // and one commit per stage.  Each wait-and-commit cycle costs the tensor pipe a fixed
    // ~0.13 us, a third of a 64-deep stage of 256 x 256 MMAs (measured without loads or
    // epilogue: gate_up forward 0.327 vs 0.373 ms with six 64-deep stages; with them the
    // step is 1-2 % faster).
    static constexpr int KB2 = (PAIR && !QB) ? 2 : 1;
    static constexpr int kSubBytes = kABytes * KW + ((kBBytes + 1023) / 1024) * 1024;   // one k-block
    static constexpr int kStageBytes = KB2 * kSubBytes;
    static constexpr int kStages = PAIR ? 6 / KB2 : (BN >= 256 ? 4 : (216 * 1024) / kStageBytes);
    static constexpr int kAccCols = BN;
    static constexpr uint32_t kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
    // NF4: the block scales of a stage's B half (128 rows of one 64-element block each) land
    // by TMA with its codes, in a slot of their own after the ring
    static constexpr int kScaleBytes = QB == 4 ? 128 * 4 : 0;
    static constexpr size_t kSmem = 1024 + (size_t)kStages * (kStageBytes + kScaleBytes) + 256;
};

struct TcParams {
    CUtensorMap tm_a, tm_b, tm_a2, tm_b2;
    CUtensorMap tm_a64, tm_a2_64;   // SM pairs: 64-row boxes of A / A2 for half tiles
    CUtensorMap tm_bs;              // NF4: block scales [E][ldb / 64][rows of B[e]] (float32)
    GroupedGemm g;
    int num_kb;         // K / 64
    int lora_k16;       // RP / 16 (0: no LoRA step)
    int n_tiles;        // output-column tiles
    int a2_bytes;       // bytes of the A2 tile
    int b2_box_bytes;   // bytes of one B2 box (64 columns x RP rows)
    uint32_t a2_sbo, a2_swz;
    uint64_t wait_ns;   // limit of the ordinary bounded waits
    int stall;          // diagnostics: the epilogue first waits on a barrier nothing arrives on
    float nf4[16];      // NF4 code values (quantised B with 4-bit codes)
};

// Tile order: expert by expert; inside an expert, bands of kRasterRows row tiles, and in a
// band the column tiles outer, the row tiles inner.  The CTAs that run at the same time then
// share each weight slab (one expert's column tile) while it is in L2, instead of every
// expert that straddles two waves of tiles loading all its slabs twice.  Each tile is
// computed the same way whatever its place in the order, so results do not depend on it.
constexpr int kRasterRows = 4;

__device__ __forceinline__ void decode_tile(int t, int n_tiles, const int32_t* s_toff, int E, int& e, int& mt,
                                            int& nt) {
    e = expert_of_row(s_toff, E, t / n_tiles);
    const int rt = s_toff[e + 1] - s_toff[e];              // row tiles of expert e (>= 1)
    const int local = t - s_toff[e] * n_tiles;
    const int band = local / (kRasterRows * n_tiles);
    const int r0 = band * kRasterRows;
    const int rows = min(kRasterRows, rt - r0);
    const int r = local - r0 * n_tiles;
    nt = r / rows;
    mt = r0 + (r - nt * rows);
}

__device__ __forceinline__ void set_timeout(const GroupedGemm& g, volatile int* s_abort) {
    *s_abort = 1;
    atomicOr(g.dev_status, MOE_DEV_TIMEOUT);
}

__device__ __forceinline__ uint4 pack8_bf16(const float* f) {
    uint4 v;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return v;
}

__device__ __forceinline__ void unpack8_bf16(const uint4& v, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

template <bool PAIRED, int BN>
__device__ __forceinline__ int b_col(int j, int nt, int ncols) {
    if (PAIRED) return (j < 2 ? 0 : ncols) + nt * (BN / 2) + (j & 1) * 64;
    return nt * BN + j * 64;
}

// SM pairs: first column of box jj (0, 1) of CTA `rank`'s half of B.  A full tile (M = 256)
// gives CTA 0 the instruction's columns [0, 128) and CTA 1 [128, 256): for gate/up pairs
// that is (gate 0-63, gate 64-127 | up 0-63, up 64-127).  A half tile (M = 128, 64 rows per
// CTA) folds the columns [128, 256) onto TMEM lanes 64-127 of the same TMEM columns, so for
// gate/up pairs it takes (gate 0-63, up 0-63 | gate 64-127, up 64-127): each epilogue thread
// then holds the gate and the up accumulator of the same output column.
template <bool PAIRED, int BN>
__device__ __forceinline__ int b_col_pair(bool half, int rank, int jj, int nt, int ncols) {
    if (PAIRED && half) return (jj == 0 ? 0 : ncols) + nt * (BN / 2) + rank * 64;
    return b_col<PAIRED, BN>(2 * rank + jj, nt, ncols);
}

// SM pairs: a tile holds 256 rows of one expert; the expert's last tile is a half tile
// (one M = 128 instruction, 64 rows per CTA) when at most 128 of its rows are left.
__device__ __forceinline__ bool half_tile(const int32_t* s_off, int e, int mt) {
    return s_off[e + 1] - (s_off[e] + mt * 2 * BM) <= BM;
}

// ---- e4m3 -> bf16 by bit placement.  A code c = s|eeee|mmm placed as the bf16 bit
// pattern s|0000eeee|mmm0000 has the value c * 2^-120 (for e = 0 too: the pattern is then
// a bf16 subnormal with the same mantissa), so one exact bf16 multiply by 2^120 * scale
// (a power of two) gives the dequantised weight.  When 2^120 * scale is beyond bf16's
// range (scale > 2^7) the multiply is split into 2^120 and scale.
constexpr uint32_t kBf16x2Pow120 = 0x7B807B80u;    // (2^120, 2^120)

// biased binary exponent of a power of two (fp32 subnormals included); -1000 for zero
__device__ __forceinline__ int pow2_biased_exp(float s) {
    const uint32_t b = __float_as_uint(s);
    const int e = (int)((b >> 23) & 0xffu);
    return e ? e : (b ? ilogbf(s) + 127 : -1000);
}

// bf16 bit pattern of the power of two with biased exponent e (subnormal below 1; 0 for none)
__device__ __forceinline__ uint32_t bf16_pow2_bits(int e) {
    return e >= 1 ? (uint32_t)e << 7 : (e >= -6 ? 1u << (e + 6) : 0u);
}

// multipliers for 8 consecutive columns (bf16x2 pairs) from their scales; sets `big` when
// 2^120 * scale overflows bf16 for one of them, and then holds the scales themselves
__device__ __forceinline__ void fp8_multipliers(const float* sc, uint32_t* m, bool& big) {
    // common case, all eight scales normal powers of two <= 2^7: the bf16 pattern of a
    // power of two is the upper half of its fp32 pattern, and 120 << 7 adds 120 to the
    // exponent field
    uint32_t b[8];
    bool fast = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        b[i] = __float_as_uint(sc[i]);
        fast &= b[i] - 0x00800000u <= 0x43000000u - 0x00800000u;
    }
    if (fast) {
        big = false;
#pragma unroll
        for (int i = 0; i < 4; ++i) m[i] = __byte_perm(b[2 * i], b[2 * i + 1], 0x7632) + 0x3C003C00u;
        return;
    }
    int e[8];
    big = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        e[i] = pow2_biased_exp(sc[i]);
        big |= e[i] + 120 > 254;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int a = e[2 * i] + (big ? 0 : 120), b = e[2 * i + 1] + (big ? 0 : 120);
        m[i] = bf16_pow2_bits(a) | (bf16_pow2_bits(b) << 16);
    }
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
    __nv_bfloat162 r = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
}

// 8 e4m3 codes (two words, first code in the low byte) -> 8 bf16 values (four words)
__device__ __forceinline__ uint4 fp8x8_to_bf16(uint2 q, const uint32_t* m, bool big) {
    uint32_t o[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t w = h ? q.y : q.x;
        const uint32_t v = __byte_perm(w, 0, 0x3120);      // lanes (c0 | c2 << 8, c1 | c3 << 8)
        o[2 * h] = ((v & 0x007f007fu) << 4) | ((v << 8) & 0x80008000u);     // (c0, c1)
        o[2 * h + 1] = ((v & 0x7f007f00u) >> 4) | (v & 0x80008000u);       // (c2, c3)
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = hmul2_bits(big ? hmul2_bits(o[i], kBf16x2Pow120) : o[i], m[i]);
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// ---- NF4 -> bf16 by selection.  The 64 codes of a row share one scale, so the row's 16
// possible values P[c] = bf16(T[c] * scale) are formed once and split into byte planes:
// lo[q] holds the low bytes of P[4q .. 4q+3], hi[q] their high bytes.  A code's two bytes
// are then picked with byte permutes: its low three bits choose one of the 8 bytes of
// each pair of plane words (codes 0-7, codes 8-15), and a third permute, steered by its
// high bit, keeps the right one of the two.
__device__ __forceinline__ void nf4_planes(const float* T, float s, uint32_t* lo, uint32_t* hi) {
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(__fmul_rn(T[2 * k], s), __fmul_rn(T[2 * k + 1], s));
        w[k] = *reinterpret_cast<const uint32_t*>(&p);           // (P[2k], P[2k+1])
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        lo[q] = __byte_perm(w[2 * q], w[2 * q + 1], 0x6420);
        hi[q] = __byte_perm(w[2 * q], w[2 * q + 1], 0x7531);
    }
}

// 8 NF4 codes (one word, the first code in the low nibble) -> 8 bf16 values (four words);
// 21 integer instructions
__device__ __forceinline__ uint4 nf4x8_to_bf16(uint32_t q, const uint32_t* lo, const uint32_t* hi) {
    const uint32_t sel = q & 0x77777777u;                          // byte within a pair of plane words
    // result byte i of a two-word permute: byte i of the first word, or of the second
    // (selector i + 4) where the code is >= 8
    const uint32_t pick = ((q >> 1) & 0x44444444u) | 0x32103210u;
    uint32_t o[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t s = h ? sel >> 16 : sel, p = h ? pick >> 16 : pick;   // codes 4h .. 4h+3
        const uint32_t l = __byte_perm(__byte_perm(lo[0], lo[1], s), __byte_perm(lo[2], lo[3], s), p);
        const uint32_t u = __byte_perm(__byte_perm(hi[0], hi[1], s), __byte_perm(hi[2], hi[3], s), p);
        o[2 * h] = __byte_perm(l, u, 0x5140);                      // (P[c0], P[c1])
        o[2 * h + 1] = __byte_perm(l, u, 0x7362);                  // (P[c2], P[c3])
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int EPI, bool B_MN, int BN, bool PAIR, int QB, int CG>
__global__ void __launch_bounds__(threads_of(CG), 1) grouped_gemm_tc_kernel(const __grid_constant__ TcParams P) {
    pdl_wait();      // no early trigger: dependents launch when this long kernel completes
    constexpr bool PAIRED = (EPI == EPI_SWIGLU);
    using G = Geo<BN, PAIR, QB>;
    constexpr bool QW = QB != 0;                    // quantised weights (e4m3 or NF4 codes)
    static_assert(QW == (CG != 0) && (CG == 0 || CG == 2 || CG == 3), "converter groups with quantised weights");
    constexpr int kEpiWarps = epi_warps(CG);
    constexpr int kConvGroups = QW ? CG : 1;       // (1 sizes the drain's per-group arrays)
    constexpr int kConvWarps = 4 * CG;
    static_assert(QB == 0 || QB == 8 || QB == 4, "e4m3 or NF4 codes");
    static_assert(!QW || BN == 256, "quantised weights are for the expert GEMMs");
    static_assert(!QW || PAIR, "quantised weights run on SM pairs (each CTA dequantises half of the B tile)");
    constexpr int kStages = G::kStages;
    constexpr int kStageBytes = G::kStageBytes;
    constexpr int kAccCols = G::kAccCols;
    constexpr uint32_t kTmemCols = G::kTmemCols;
    constexpr int TM = PAIR ? 2 * BM : BM;          // rows per tile
    static_assert(BN == 256 || !B_MN, "narrow tiles take a K-major B");
    static_assert(!PAIR || BN == 256, "SM pairs run the 256-wide expert GEMMs only");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* s_scale = reinterpret_cast<float*>(smem + kStages * kStageBytes);   // NF4: kStages x 128 scales
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kStages * (kStageBytes + G::kScaleBytes));
    uint64_t* empty_bar = full_bar + kStages;
    uint64_t* tfull_bar = empty_bar + kStages;
    uint64_t* tempty_bar = tfull_bar + 2;
    uint64_t* staged_bar = tempty_bar + 2;          // quantised B: codes (and NF4 scales) landed
    uint64_t* drain_bar = staged_bar + kStages;     // after an abort: the MMA issuer's last commit
    uint64_t* stall_bar = drain_bar + 1;            // diagnostics: nothing ever arrives on it
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stall_bar + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint32_t* sig_slot = tmem_slot + 2;             // quantised pairs: target of the peer's stage signals
    // what the roles issued, read by the abort drain: [0] the producer's stage fills,
    // [1 + g] the stages converter group g signalled (quantised B); [kDebugSlot] debug
    // build: bad offsets
    volatile int* s_issued = reinterpret_cast<volatile int*>(tmem_slot + 4);
    constexpr int kDebugSlot = 1 + kConvGroups;
    int32_t* s_off = reinterpret_cast<int32_t*>(tmem_slot + 12);
    static_assert(4 + kDebugSlot < 12, "issue counters fit before the offsets");
    static_assert((3 * kStages + 6) * 8 + 48 <= 256, "barriers and flags fit the 256-byte tail");
    const GroupedGemm& g = P.g;
    const int E = g.E;
    int32_t* s_toff = s_off + (E + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? tc::cluster_rank() : 0u;     // 0 = leader of the pair
    const int tile0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int tile_step = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

    for (int i = threadIdx.x; i <= E; i += blockDim.x) {
        s_off[i] = g.offsets[i];
        if (!PAIR) s_toff[i] = g.tile_offsets[i];
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            // with quantised weights the B half of a stage is complete when the converter group
            // that owns the stage has arrived (and, in a pair, the peer's group has completed
            // kSignalBytes transaction bytes on it)
            tc::mbar_init(tc::smem_u32(&full_bar[s]), QW ? 2 : 1);
            tc::mbar_init(tc::smem_u32(&empty_bar[s]), 1);
            tc::mbar_init(tc::smem_u32(&staged_bar[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(tc::smem_u32(&tfull_bar[a]), 1);
            tc::mbar_init(tc::smem_u32(&tempty_bar[a]), PAIR ? 2 * kEpiWarps : kEpiWarps);
        }
        tc::mbar_init(tc::smem_u32(drain_bar), 1);
        tc::mbar_init(tc::smem_u32(stall_bar), 1);
        *s_abort = 0;
        for (int i = 0; i < 1 + kConvGroups; ++i) s_issued[i] = 0;
        tc::fence_mbar_init();
    }
    if constexpr (PAIR) {
        // 256-row tile offsets: prefix sum of ceil(count / 256) (warp 0, 32 experts per step)
        __syncthreads();
        if (warp == 0) {
            int run = 0;
            for (int b = 0; b < E; b += 32) {
                const int e = b + lane;
                const int v = e < E ? (s_off[e + 1] - s_off[e] + TM - 1) / TM : 0;
                int incl = v;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int n = __shfl_up_sync(0xffffffffu, incl, d);
                    if (lane >= d) incl += n;
                }
                if (e < E) s_toff[e] = run + incl - v;
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) s_toff[E] = run;
        }
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&P.tm_a);
        tc::prefetch_tmap(&P.tm_b);
        if (PAIR) tc::prefetch_tmap(&P.tm_a64);
        if (QB == 4) tc::prefetch_tmap(&P.tm_bs);
        if (P.lora_k16) {
            tc::prefetch_tmap(&P.tm_a2);
            tc::prefetch_tmap(&P.tm_b2);
            if (PAIR) tc::prefetch_tmap(&P.tm_a2_64);
        }
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tc::tmem_alloc_pair(tc::smem_u32(tmem_slot), kTmemCols);
            tc::tmem_relinquish_pair();
        } else {
            tc::tmem_alloc(tc::smem_u32(tmem_slot), kTmemCols);
            tc::tmem_relinquish();
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if constexpr (PAIR) tc::cluster_sync();    // the peer's barriers exist before anyone signals them
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    if constexpr (MOE_DEBUG) {
        // debug build: offsets that do not describe N rows schedule no tile
        if (threadIdx.x == 0)
            s_issued[kDebugSlot] = dbg_offsets_ok(s_off, PAIR ? nullptr : s_toff, E, g.N, BM, g.dev_status) ? 0 : 1;
        __syncthreads();
    }
    const int total_tiles = (MOE_DEBUG && s_issued[kDebugSlot]) ? 0 : s_toff[E] * P.n_tiles;
    const uint64_t lim = P.wait_ns;
    int fills = 0;                                  // the producer's stage fills (lane 0 of warp 0)
    constexpr int KB2 = G::KB2;                     // 64-deep k-blocks per ring stage
    const int nmain = (P.num_kb + KB2 - 1) / KB2;   // main-product stages per tile (then the LoRA step)

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int t = tile0; t < total_tiles && !*s_abort; t += tile_step) {
                int e, mt, nt;
                decode_tile(t, P.n_tiles, s_toff, E, e, mt, nt);
                const bool half = PAIR && half_tile(s_off, e, mt);
                const int m0 = s_off[e] + mt * TM + (int)rank * (half ? BM / 2 : BM);   // this CTA's rows
                const CUtensorMap* tma = half ? &P.tm_a64 : &P.tm_a;
                const CUtensorMap* tma2 = half ? &P.tm_a2_64 : &P.tm_a2;
                const int a_bytes = half ? kABytes / 2 : kABytes;
                const int a2_bytes = half ? P.a2_bytes / 2 : P.a2_bytes;
                const int nkb = G::KW > 1 ? (P.num_kb + G::KW - 1) / G::KW : nmain + (P.lora_k16 ? 1 : 0);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!tc::mbar_wait(tc::smem_u32(&empty_bar[stage]), phase ^ 1, lim)) {
                        set_timeout(g, s_abort);
                        break;
                    }
                    const uint32_t fb_local = tc::smem_u32(&full_bar[stage]);
                    const uint32_t sa = tc::smem_u32(smem + stage * kStageBytes);
                    const uint32_t sb = sa + kABytes;
                    if constexpr (PAIR) {
                        // both CTAs' loads complete on the leader's full barrier
                        const uint32_t fb = tc::mapa(fb_local, 0);
                        if (kb < nmain && QW) {
                            if (rank == 0) tc::mbar_arrive_expect_tx(fb_local, 2 * a_bytes + kSignalBytes);
                            tc::tma_load_2d_pair(sa, tma, fb, kb * BK, m0);
                            // the codes land at the top of the B slot, plain rows of 64 codes
                            // (64 bytes e4m3, 32 bytes NF4); a code row's byte coordinate is its
                            // element coordinate * QB / 8
                            const uint32_t sq = sb + G::kBBytes - G::kQBytes;
                            const uint32_t qb = tc::smem_u32(&staged_bar[stage]);
                            // NF4: the stage's block scales come with its codes, on the same barrier
                            const uint32_t ss = tc::smem_u32(s_scale + stage * 128);
                            tc::mbar_arrive_expect_tx(qb, G::kQBytes + G::kScaleBytes);
                            if (B_MN) {
#pragma unroll
                                for (int jj = 0; jj < 2; ++jj) {
                                    const int col = b_col_pair<PAIRED, BN>(half, (int)rank, jj, nt, g.Ncols);
                                    tc::tma_load_3d(sq + jj * (kBoxMN * QB / 16), &P.tm_b, qb, col * QB / 8, kb * BK, e);
                                    // 64 k rows of the box's column block (a block past B[e]'s columns reads zeros)
                                    if (QB == 4) tc::tma_load_3d(ss + jj * 256, &P.tm_bs, qb, kb * BK, col / 64, e);
                                }
                            } else {
                                const int n0 = nt * BN + (int)rank * (BN / 2);
                                tc::tma_load_3d(sq, &P.tm_b, qb, kb * BK * QB / 8, n0, e);
                                // 128 n rows of the stage's k block (rows past B[e] read zeros)
                                if (QB == 4) tc::tma_load_3d(ss, &P.tm_bs, qb, n0, kb, e);
                            }
                        } else if (kb < nmain) {
                            // k-blocks kb * KB2 .. of this stage, each in its own A + B sub-block
                            const int nsub = min(KB2, P.num_kb - kb * KB2);
                            if (rank == 0) tc::mbar_arrive_expect_tx(fb_local, 2 * nsub * (a_bytes + G::kBBytes));
                            for (int j = 0; j < nsub; ++j) {
                                const uint32_t saj = sa + j * G::kSubBytes, sbj = saj + kABytes;
                                const int kx = (kb * KB2 + j) * BK;
                                tc::tma_load_2d_pair(saj, tma, fb, kx, m0);
                                if (B_MN) {
#pragma unroll
                                    for (int jj = 0; jj < 2; ++jj)
                                        tc::tma_load_3d_pair(sbj + jj * kBoxMN, &P.tm_b, fb,
                                                             b_col_pair<PAIRED, BN>(half, (int)rank, jj, nt, g.Ncols), kx, e);
                                } else {
                                    tc::tma_load_3d_pair(sbj, &P.tm_b, fb, kx, nt * BN + (int)rank * (BN / 2), e);
                                }
                            }
                        } else {
                            if (rank == 0) {
                                tc::mbar_arrive_expect_tx(fb_local, 2 * (a2_bytes + 2 * P.b2_box_bytes));
                                // quantised B: the LoRA step needs no conversion; the producer makes both arrivals
                                if (QW) tc::mbar_arrive(fb_local);
                            }
                            tc::tma_load_2d_pair(sa, tma2, fb, 0, m0);
#pragma unroll
                            for (int jj = 0; jj < 2; ++jj)
                                tc::tma_load_3d_pair(sb + jj * P.b2_box_bytes, &P.tm_b2, fb,
                                                     b_col_pair<PAIRED, BN>(half, (int)rank, jj, nt, g.Ncols), 0, e);
                        }
                    } else if constexpr (G::KW > 1) {
                        // narrow tile: KW consecutive 64-column boxes of A and of B per stage
                        const uint32_t fb = fb_local;
                        const int nbox = min(G::KW, P.num_kb - kb * G::KW);
                        tc::mbar_arrive_expect_tx(fb, nbox * (kABytes + BN * BK * 2));
                        for (int j = 0; j < nbox; ++j) {
                            const int kx = (kb * G::KW + j) * BK;
                            tc::tma_load_2d(sa + j * kABytes, &P.tm_a, fb, kx, m0);
                            tc::tma_load_3d(sa + G::KW * kABytes + j * (BN * BK * 2), &P.tm_b, fb, kx, nt * BN, e);
                        }
                    } else {
                        // single-CTA tile (bf16 weights only)
                        const uint32_t fb = fb_local;
                        if (kb < nmain) {
                            tc::mbar_arrive_expect_tx(fb, kABytes + G::kBBytes);
                            tc::tma_load_2d(sa, &P.tm_a, fb, kb * BK, m0);
                            if (B_MN) {
#pragma unroll
                                for (int j = 0; j < 4; ++j)
                                    tc::tma_load_3d(sb + j * kBoxMN, &P.tm_b, fb, b_col<PAIRED, BN>(j, nt, g.Ncols),
                                                    kb * BK, e);
                            } else {
                                tc::tma_load_3d(sb, &P.tm_b, fb, kb * BK, nt * BN, e);
                            }
                        } else {
                            tc::mbar_arrive_expect_tx(fb, P.a2_bytes + 4 * P.b2_box_bytes);
                            tc::tma_load_2d(sa, &P.tm_a2, fb, 0, m0);
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                tc::tma_load_3d(sb + j * P.b2_box_bytes, &P.tm_b2, fb, b_col<PAIRED, BN>(j, nt, g.Ncols),
                                                0, e);
                        }
                    }
                    ++fills;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            s_issued[0] = fills;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader only for pairs)
        if (lane == 0 && rank == 0) {
            const uint32_t idesc_full = tc::idesc_bf16(TM, BN, false, B_MN);
            const uint32_t idesc2_full = tc::idesc_bf16(TM, BN, false, true);
            // SM pairs, half tile: M = 128 (64 rows per CTA)
            const uint32_t idesc_half = tc::idesc_bf16(BM, BN, false, B_MN);
            const uint32_t idesc2_half = tc::idesc_bf16(BM, BN, false, true);
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            for (int t = tile0; t < total_tiles && !*s_abort; t += tile_step, ++it) {
                const int acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!tc::mbar_wait(tc::smem_u32(&tempty_bar[acc]), acc_phase ^ 1, lim)) {
                    set_timeout(g, s_abort);
                    break;
                }
                tc::fence_after_sync();
                const uint32_t d = tmem_base + acc * kAccCols;
                bool half = false;
                if constexpr (PAIR) {
                    int e, mt, nt;
                    decode_tile(t, P.n_tiles, s_toff, E, e, mt, nt);
                    half = half_tile(s_off, e, mt);
                }
                const uint32_t idesc = half ? idesc_half : idesc_full;
                const uint32_t idesc2 = half ? idesc2_half : idesc2_full;
                const int nkb = G::KW > 1 ? (P.num_kb + G::KW - 1) / G::KW : nmain + (P.lora_k16 ? 1 : 0);
                bool ok = true;
                for (int kb = 0; kb < nkb; ++kb) {
                    // quantised pairs: the peer's converted half is published by a cluster-scope release
                    if (!tc::mbar_wait<QW && PAIR>(tc::smem_u32(&full_bar[stage]), phase, lim)) {
                        set_timeout(g, s_abort);
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t sa = tc::smem_u32(smem + stage * kStageBytes);
                    const uint32_t sb = sa + kABytes;
                    if constexpr (G::KW > 1) {
                        const int nbox = min(G::KW, P.num_kb - kb * G::KW);
                        for (int j = 0; j < nbox; ++j) {
#pragma unroll
                            for (int kk = 0; kk < BK / 16; ++kk) {
                                const uint64_t ad = tc::smem_desc(sa + j * kABytes + kk * 32, 16, 1024, tc::kSw128);
                                const uint64_t bd = tc::smem_desc(sa + G::KW * kABytes + j * (BN * BK * 2) + kk * 32, 16,
                                                                  1024, tc::kSw128);
                                tc::mma_bf16(d, ad, bd, idesc, (kb > 0 || j > 0 || kk > 0) ? 1u : 0u);
                            }
                        }
                    } else if (kb < nmain) {
                        const int nsub = min(KB2, P.num_kb - kb * KB2);
#pragma unroll
                        for (int j = 0; j < KB2; ++j) {
                            if (j >= nsub) break;
                            const uint32_t saj = sa + j * G::kSubBytes, sbj = saj + kABytes;
#pragma unroll
                            for (int kk = 0; kk < BK / 16; ++kk) {
                                const uint64_t ad = tc::smem_desc(saj + kk * 32, 16, 1024, tc::kSw128);
                                const uint64_t bd = B_MN ? tc::smem_desc(sbj + kk * 2048, kBoxMN, 1024, tc::kSw128)
                                                         : tc::smem_desc(sbj + kk * 32, 16, 1024, tc::kSw128);
                                const uint32_t acc_in = (kb > 0 || j > 0 || kk > 0) ? 1u : 0u;
                                if constexpr (PAIR) tc::mma_bf16_pair(d, ad, bd, idesc, acc_in);
                                else tc::mma_bf16(d, ad, bd, idesc, acc_in);
                            }
                        }
                    } else {
                        for (int kk = 0; kk < P.lora_k16; ++kk) {
                            const uint64_t ad = tc::smem_desc(sa + kk * 32, 16, P.a2_sbo, P.a2_swz);
                            const uint64_t bd = tc::smem_desc(sb + kk * 2048, P.b2_box_bytes, 1024, tc::kSw128);
                            if constexpr (PAIR) tc::mma_bf16_pair(d, ad, bd, idesc2, 1u);
                            else tc::mma_bf16(d, ad, bd, idesc2, 1u);
                        }
                    }
                    if constexpr (PAIR) tc::mma_commit_pair(tc::smem_u32(&empty_bar[stage]), 0x3);
                    else tc::mma_commit(tc::smem_u32(&empty_bar[stage]));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                if constexpr (PAIR) tc::mma_commit_pair(tc::smem_u32(&tfull_bar[acc]), 0x3);
                else tc::mma_commit(tc::smem_u32(&tfull_bar[acc]));
            }
        }
    } else if (QW && warp >= 2 + kEpiWarps) {
        // ------------------------------------------------------------ dequantisers
        // codes (staging slot, plain row-major boxes of 64 codes per row) -> bf16 in the
        // 128-byte-swizzled layout TMA would have written: row r, 16-byte chunk cc of 8
        // elements at r * 128 + ((cc ^ (r & 7)) << 4).  e4m3: each value times its column's
        // power-of-two scale (exact, fp8x8_to_bf16).
        if constexpr (QB == 8) {
            constexpr int kGT = 32 * (kConvWarps / kConvGroups);    // threads of one group
            constexpr int kUnits = G::kQBytes / 8;                  // 8 codes per unit
            constexpr int kIters = kUnits / kGT;
            constexpr int kBoxes = B_MN ? 2 : 1;                   // 64-column code boxes per CTA (SM pairs)
            static_assert(kUnits % kGT == 0 && 512 % kGT == 0, "units per stage must split evenly");
            static_assert(kStages % kConvGroups == 0, "every group owns whole stages");
            const int ct = threadIdx.x - 32 * (2 + kEpiWarps);
            const int grp = ct / kGT;
            const int gt = ct % kGT;
            const int cc = gt & 7;                                  // the thread's 16-byte chunk of a row
            const uint32_t full_leader0 = tc::mapa(tc::smem_u32(&full_bar[0]), 0);
            const uint32_t sig_leader = tc::mapa(tc::smem_u32(sig_slot), 0);
            int stage = 0;
            uint32_t sbits = 0;                                     // per-stage parity of staged_bar
            int done = 0;                                           // stages this group has signalled
            bool ok = true;
            uint32_t fm[kBoxes][4];                                 // multipliers of this thread's chunks
            bool big[kBoxes];
            // the warps of a group leave together: every exit decision is a group-wide vote
            // (an abort elsewhere stops the producer, and the next staged wait then runs out)
            for (int t = tile0; t < total_tiles && ok; t += tile_step) {
                int e, mt, nt;
                decode_tile(t, P.n_tiles, s_toff, E, e, mt, nt);
                const float* se = g.b_scale + (int64_t)e * g.ldb;
                if constexpr (B_MN) {
                    // MN-major: a chunk's scales depend on its columns only, fixed for the tile
#pragma unroll
                    for (int j = 0; j < kBoxes; ++j) {
                        const int col = b_col_pair<PAIRED, BN>(half_tile(s_off, e, mt), (int)rank, j, nt, g.Ncols) + cc * 8;
                        const bool in = col < g.ldb;
                        const float4 a = in ? __ldg(reinterpret_cast<const float4*>(se + col)) : make_float4(0, 0, 0, 0);
                        const float4 b = in ? __ldg(reinterpret_cast<const float4*>(se + col) + 1) : make_float4(0, 0, 0, 0);
                        const float sc[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                        fp8_multipliers(sc, fm[j], big[j]);
                    }
                }
                const int nkb = P.num_kb + (P.lora_k16 ? 1 : 0);
                for (int kb = 0; kb < nkb; ++kb) {
                    const bool mine = (stage % kConvGroups) == grp;
                    if (mine && kb < P.num_kb) {
                        // K-major: the scales follow k; loaded before the wait, used after it
                        float4 ka, kb4;
                        if constexpr (!B_MN) {
                            ka = __ldg(reinterpret_cast<const float4*>(se + kb * BK + cc * 8));
                            kb4 = __ldg(reinterpret_cast<const float4*>(se + kb * BK + cc * 8) + 1);
                        }
                        const bool got = tc::mbar_wait(tc::smem_u32(&staged_bar[stage]), (sbits >> stage) & 1u, lim);
                        if (!tc::named_bar_and(1 + grp, kGT, got && !*s_abort)) {
                            if (gt == 0) set_timeout(g, s_abort);
                            ok = false;
                            break;
                        }
                        sbits ^= 1u << stage;
                        if constexpr (!B_MN) {
                            const float sc[8] = {ka.x, ka.y, ka.z, ka.w, kb4.x, kb4.y, kb4.z, kb4.w};
                            fp8_multipliers(sc, fm[0], big[0]);
                        }
                        uint8_t* bt = smem + stage * kStageBytes + kABytes;
                        const uint8_t* qt = bt + G::kBBytes - G::kQBytes;
                        // all of the group's codes are read before any bf16 value overwrites them
                        uint2 q[kIters];
#pragma unroll
                        for (int i = 0; i < kIters; ++i) {
                            const int u = gt + kGT * i;
                            const int j = B_MN ? (i * kGT) / 512 : 0;   // gt < kGT and kGT divides 512
                            const int r = B_MN ? ((u >> 3) & 63) : (u >> 3);
                            q[i] = *reinterpret_cast<const uint2*>(qt + j * (kBoxMN / 2) + r * 64 + cc * 8);
                        }
                        tc::named_bar_sync(1 + grp, kGT);
#pragma unroll
                        for (int i = 0; i < kIters; ++i) {
                            const int u = gt + kGT * i;
                            const int j = B_MN ? (i * kGT) / 512 : 0;
                            const int r = B_MN ? ((u >> 3) & 63) : (u >> 3);
                            *reinterpret_cast<uint4*>(bt + j * kBoxMN + r * 128 + ((cc ^ (r & 7)) << 4)) =
                                fp8x8_to_bf16(q[i], fm[j], big[j]);
                        }
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    }
                    if (mine && kb < P.num_kb) {
                        // one signal per group and converted stage, after every thread's writes and
                        // proxy fence: a CTA-scope arrive on this CTA's full barrier, or from the peer
                        // of a pair an asynchronous store that completes transaction bytes on the
                        // leader's (a cluster-scope arrive would hold the thread for a microsecond).
                        // The LoRA step is not converted: its producer makes both arrivals, after its
                        // wait for the stage to be free, so no arrival can reach an earlier phase.
                        tc::named_bar_sync(1 + grp, kGT);
                        if (gt == 0) {
                            if (rank == 0) tc::mbar_arrive(tc::smem_u32(&full_bar[stage]));
                            else tc::st_async_signal(sig_leader, 1u, full_leader0 + stage * (uint32_t)sizeof(uint64_t));
                        }
                        ++done;
                    }
                    if (++stage == kStages) stage = 0;
                }
            }
            if (gt == 0) s_issued[1 + grp] = done;
        } else if constexpr (QB == 4) {
            // NF4: plain rows of 32 bytes (64 codes, two per byte, the even element in the
            // low nibble) -> bf16(T[code] * absmax).  One thread per B row of the stage (64 k
            // rows x 2 boxes of an MN-major B, 128 n rows of a K-major B); each such row is
            // one 64-element block with one scale, so the thread forms its 16 possible values
            // once and then only selects among them (nf4x8_to_bf16).  Stage ownership,
            // barriers and the signal are those of the e4m3 converter.
            constexpr int kGT = 32 * (kConvWarps / kConvGroups);    // threads of one group
            static_assert(kGT == 128 && G::kQBytes == 128 * 32, "one 32-byte code row per converter thread");
            static_assert(kStages % kConvGroups == 0, "every group owns whole stages");
            const int ct = threadIdx.x - 32 * (2 + kEpiWarps);
            const int grp = ct / kGT;
            const int gt = ct % kGT;
            const int jb = B_MN ? gt >> 6 : 0;                      // MN-major: the thread's 64-column box
            const int r = B_MN ? gt & 63 : gt;                      // its row: k in the box, or n in the tile
            const uint32_t full_leader0 = tc::mapa(tc::smem_u32(&full_bar[0]), 0);
            const uint32_t sig_leader = tc::mapa(tc::smem_u32(sig_slot), 0);
            int stage = 0;
            uint32_t sbits = 0;                                     // per-stage parity of staged_bar
            int done = 0;                                           // stages this group has signalled
            bool ok = true;
            for (int t = tile0; t < total_tiles && ok; t += tile_step) {
                const int nkb = P.num_kb + (P.lora_k16 ? 1 : 0);
                for (int kb = 0; kb < nkb; ++kb) {
                    const bool mine = (stage % kConvGroups) == grp;
                    if (mine && kb < P.num_kb) {
                        const bool got = tc::mbar_wait(tc::smem_u32(&staged_bar[stage]), (sbits >> stage) & 1u, lim);
                        if (!tc::named_bar_and(1 + grp, kGT, got && !*s_abort)) {
                            if (gt == 0) set_timeout(g, s_abort);
                            ok = false;
                            break;
                        }
                        sbits ^= 1u << stage;
                        uint8_t* bt = smem + stage * kStageBytes + kABytes;
                        const uint4* qrow = reinterpret_cast<const uint4*>(bt + G::kBBytes - G::kQBytes + jb * 2048 + r * 32);
                        const uint4 q0 = qrow[0], q1 = qrow[1];
                        // the row's scale landed with the codes: MN-major, k row r of box jb's
                        // column block; K-major, n row r in the stage's k block
                        const float sc = s_scale[stage * 128 + jb * 64 + r];
                        uint32_t lo[4], hi[4];
                        nf4_planes(P.nf4, sc, lo, hi);
                        // all of the group's codes are read before any bf16 value overwrites them
                        tc::named_bar_sync(1 + grp, kGT);
                        uint8_t* row = bt + jb * kBoxMN + r * 128;
                        const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                        for (int cc = 0; cc < 8; ++cc)
                            *reinterpret_cast<uint4*>(row + ((cc ^ (r & 7)) << 4)) = nf4x8_to_bf16(qw[cc], lo, hi);
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        // one signal per group and converted stage, as in the e4m3 converter
                        tc::named_bar_sync(1 + grp, kGT);
                        if (gt == 0) {
                            if (rank == 0) tc::mbar_arrive(tc::smem_u32(&full_bar[stage]));
                            else tc::st_async_signal(sig_leader, 1u, full_leader0 + stage * (uint32_t)sizeof(uint64_t));
                        }
                        ++done;
                    }
                    if (++stage == kStages) stage = 0;
                }
            }
            if (gt == 0) s_issued[1 + grp] = done;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // warp w reads TMEM lanes 32*(w%4)..+31 (one row per thread); with 8 epilogue warps
        // the two warps of a lane quarter split the columns in halves, with 4 one warp takes
        // them all.  Half tiles (SM pairs, M = 128): lane L holds row L mod 64, lanes 64-127
        // the upper half of the columns in the same TMEM columns, so each warp covers half as
        // many TMEM columns.
        const int q = warp & 3;
        const int hw = (warp - 2) >> 2;                                 // 0 with 4 epilogue warps
        const int row = q * 32 + lane;
        constexpr int kSpan = (PAIRED ? BN / 4 : (BN >= 32 ? BN / 2 : BN)) * (8 / kEpiWarps);   // columns per warp
        const int c0 = (BN >= 32 || PAIRED) ? hw * kSpan : 0;
        const bool active = (BN >= 32 || PAIRED) || hw == 0;
        int it = 0;
        const uint32_t tempty_leader0 = PAIR ? tc::mapa(tc::smem_u32(&tempty_bar[0]), 0) : 0u;
        for (int t = tile0; t < total_tiles; t += tile_step, ++it) {
            int e, mt, nt;
            decode_tile(t, P.n_tiles, s_toff, E, e, mt, nt);
            const bool htile = PAIR && half_tile(s_off, e, mt);
            const int m0 = s_off[e] + mt * TM + (int)rank * (htile ? BM / 2 : BM);
            const int row_end = s_off[e + 1];
            const int span = htile ? kSpan / 2 : kSpan;                 // TMEM columns of this warp
            // Store pacing: all CTAs reach tile boundaries together, and their epilogue store
            // bursts slow the next tile's first TMA loads.  While the CTA has another tile
            // queued (the MMAs are busy with it, and this accumulator is not needed before the
            // tile after that) the plain-store epilogues spread their chunks 0.5 us apart
            // (measured: 2-10 % faster gate_up backward and down forward).
            const bool pace = EPI == EPI_BF16 && t + tile_step < total_tiles;
            const int cb0 = htile ? hw * span : c0;
            const int nbase = htile ? (q >> 1) * (PAIRED ? BN / 4 : BN / 2) : 0;   // output column offset
            const int up_off = htile ? BN / 4 : BN / 2;                 // gate/up pairs: up's TMEM column - gate's
            const int acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            // diagnostics: a launch chosen to fail first waits on a barrier nothing arrives on
            const bool ok = (P.stall == 0 || tc::mbar_wait(tc::smem_u32(stall_bar), 0, lim)) &&
                            tc::mbar_wait(tc::smem_u32(&tfull_bar[acc]), acc_phase, lim);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) set_timeout(g, s_abort);
                break;
            }
            tc::fence_after_sync();
            const uint32_t tb = tmem_base + acc * kAccCols + ((uint32_t)(q * 32) << 16);
            const int p = m0 + (htile ? (row & 63) : row);
            const bool valid = p < row_end;
            if (!active) {
            } else if constexpr (EPI == EPI_SWIGLU) {
                const int I = g.Ncols;
                bf16* GU = (bf16*)g.out0;
                bf16* Hh = (bf16*)g.out1;
#pragma unroll 1
                for (int c = cb0; c < cb0 + span; c += 16) {
                    float gv[16], uv[16];
                    tc::tmem_ld16(tb + c, gv);
                    tc::tmem_ld16(tb + up_off + c, uv);
                    tc::tmem_ld_wait();
                    const int n = nt * (BN / 2) + nbase + c;
                    if (valid && n < I) {
                        const uint4 g0 = pack8_bf16(gv), g1 = pack8_bf16(gv + 8);
                        const uint4 u0 = pack8_bf16(uv), u1 = pack8_bf16(uv + 8);
                        if (g.h_from_gu) {
                            // h from the stored (bf16) gate and up values, so that
                            // swiglu_rows rebuilds it bit for bit from GU alone
                            unpack8_bf16(g0, gv);
                            unpack8_bf16(g1, gv + 8);
                            unpack8_bf16(u0, uv);
                            unpack8_bf16(u1, uv + 8);
                        }
                        float hv[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) hv[i] = swiglu_f(gv[i], uv[i]);
                        // one full 32-byte sector per thread and store; GU is only read again
                        // by the backward: stream it past L2 (evict-first)
                        tc::st32_cs(GU + (int64_t)p * 2 * I + n, g0, g1);
                        tc::st32_cs(GU + (int64_t)p * 2 * I + I + n, u0, u1);
                        tc::st32(Hh + (int64_t)p * I + n, pack8_bf16(hv), pack8_bf16(hv + 8));
                    }
                }
            } else if constexpr (EPI == EPI_DSWIGLU) {
                const int I = g.Ncols;
                const bf16* GU = (const bf16*)g.gu_in;
                bf16* dGU = (bf16*)g.out0;
                const bf16* grow = GU + (int64_t)p * 2 * I;
                // prefetch the (g, u) pair of the next 16 columns while this chunk computes
                uint4 pg0 = make_uint4(0, 0, 0, 0), pg1 = pg0, pu0 = pg0, pu1 = pg0;
                {
                    const int n = nt * BN + nbase + cb0;
                    if (valid && n < I) {
                        tc::ld32_nc(grow + n, pg0, pg1);
                        tc::ld32_nc(grow + I + n, pu0, pu1);
                    }
                }
#pragma unroll 1
                for (int c = cb0; c < cb0 + span; c += 16) {
                    const uint4 g0 = pg0, g1 = pg1, u0 = pu0, u1 = pu1;
                    const int n = nt * BN + nbase + c;
                    const int nn = n + 16;
                    if (c + 16 < cb0 + span && valid && nn < I) {
                        tc::ld32_nc(grow + nn, pg0, pg1);
                        tc::ld32_nc(grow + I + nn, pu0, pu1);
                    }
                    float dh[16];
                    tc::tmem_ld16(tb + c, dh);
                    tc::tmem_ld_wait();
                    if (valid && n < I) {
                        float gg[16], uu[16], dg[16], du[16];
                        unpack8_bf16(g0, gg); unpack8_bf16(g1, gg + 8);
                        unpack8_bf16(u0, uu); unpack8_bf16(u1, uu + 8);
#pragma unroll
                        for (int i = 0; i < 16; ++i) dswiglu_f(dh[i], gg[i], uu[i], dg[i], du[i]);
                        tc::st32(dGU + (int64_t)p * 2 * I + n, pack8_bf16(dg), pack8_bf16(dg + 8));
                        tc::st32(dGU + (int64_t)p * 2 * I + I + n, pack8_bf16(du), pack8_bf16(du + 8));
                    }
                }
            } else if constexpr (EPI == EPI_PROJ) {
                bf16* out = (bf16*)g.out0;
#pragma unroll
                for (int c = cb0; c < cb0 + span; c += 16) {
                    float v[16];
                    tc::tmem_ld16(tb + c, v);
                    tc::tmem_ld_wait();
                    if (valid) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] *= g.scale;
                        tc::st32(out + (int64_t)p * BN + c, pack8_bf16(v), pack8_bf16(v + 8));
                    }
                }
            } else if constexpr (EPI == EPI_BF16) {
                bf16* out = (bf16*)g.out0;
#pragma unroll 1
                for (int c = cb0; c < cb0 + span; c += 16) {
                    if (pace && c != cb0) __nanosleep(kPaceNs);
                    float v[16];
                    tc::tmem_ld16(tb + c, v);
                    tc::tmem_ld_wait();
                    const int n = nt * BN + nbase + c;
                    if (valid && n < g.Ncols) {
                        // read once by the combine and once by the backward: evict-first
                        tc::st32_cs(out + (int64_t)p * g.ldo + n, pack8_bf16(v), pack8_bf16(v + 8));
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR) tc::mbar_arrive_cluster(tempty_leader0 + acc * (uint32_t)sizeof(uint64_t));
                else tc::mbar_arrive(tc::smem_u32(&tempty_bar[acc]));
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if constexpr (PAIR) tc::cluster_sync();    // normally: the leader's MMAs into the peer's TMEM are done
    // ---- abort drain.  After a wait gave up, copies and MMAs may still be in flight: loads
    // of stages nobody consumed, a pair's loads and stage signals towards the leader's full
    // barriers, MMAs of tiles whose accumulators nobody read.  Every one of them has landed
    // before the shared memory and TMEM are released: each producer waits for its own code
    // stages (quantised B), the leader completes on behalf of the side that issued nothing every
    // full-barrier phase that received any copy and waits for it, and the MMA issuer waits
    // for a last commit.  These waits use the full limit.  Both CTAs of a pair read both
    // abort flags, so they take the branch together.
    bool aborted = *s_abort != 0;
    if constexpr (PAIR)
        aborted = aborted || tc::ld_shared_cluster(tc::mapa(tc::smem_u32((const void*)s_abort), rank ^ 1u)) != 0;
    if (aborted) {
        if (warp == 0 && lane == 0) {
            // stage fills issued by each producer, stages signalled by each converter group
            const int own_f = s_issued[0];
            int peer_f = 0, peer_done[kConvGroups] = {};
            if constexpr (PAIR) {
                const uint32_t pv = tc::mapa(tc::smem_u32((const void*)s_issued), rank ^ 1u);
                peer_f = (int)tc::ld_shared_cluster(pv);
                for (int i = 0; i < kConvGroups; ++i) peer_done[i] = (int)tc::ld_shared_cluster(pv + 4u * (1 + i));
            }
            const int f_lead = rank == 0 ? own_f : peer_f, f_peer = rank == 0 ? peer_f : own_f;
            const int f_max = PAIR ? max(own_f, peer_f) : own_f;
            // The producers run at most kStages fills apart (each waits for the MMA to have
            // consumed the stage's previous fill), and every fill before f_max - kStages was
            // consumed, so its phases are complete; the fills after it are the current
            // phases of their stages.  Replay the fill sequence to find their sizes.
            const int w0 = max(0, f_max - kStages);
            int f = 0;
            uint32_t sbits = 0;
            int gcount[kConvGroups] = {};
            for (int t = tile0; t < total_tiles && f < f_max; t += tile_step) {
                int e, mt, nt;
                decode_tile(t, P.n_tiles, s_toff, E, e, mt, nt);
                const bool half = PAIR && half_tile(s_off, e, mt);
                const int nkb = G::KW > 1 ? (P.num_kb + G::KW - 1) / G::KW : nmain + (P.lora_k16 ? 1 : 0);
                for (int kb = 0; kb < nkb && f < f_max; ++kb, ++f) {
                    const int st = f % kStages;
                    const bool main = G::KW > 1 || kb < nmain;        // not the LoRA step
                    const uint32_t spar = (sbits >> st) & 1u;
                    int gi = 0;                                       // index among its group's code stages
                    if (QW && main) {
                        sbits ^= 1u << st;
                        gi = gcount[st % kConvGroups]++;
                    }
                    if (f < w0) continue;
                    if (QW && main && f < own_f) tc::mbar_wait(tc::smem_u32(&staged_bar[st]), spar);
                    if (rank != 0) continue;
                    // bytes that one CTA's copies of this fill complete on the full barrier
                    uint32_t b;
                    if (G::KW > 1) b = min(G::KW, P.num_kb - kb * G::KW) * (kABytes + BN * BK * 2);
                    else if (main) b = ((half ? kABytes / 2 : kABytes) + (QW ? 0 : G::kBBytes)) * min(KB2, P.num_kb - kb * KB2);
                    else b = (half ? P.a2_bytes / 2 : P.a2_bytes) + (PAIR ? 2 : 4) * P.b2_box_bytes;
                    const bool lp = f < f_lead, pp = PAIR && f < f_peer;
                    if (!lp && !pp) continue;                         // no copy went towards this phase
                    const int grp = st % kConvGroups;
                    const bool lc = QW && main && gi < s_issued[1 + grp];
                    const bool ps = QW && PAIR && main && gi < peer_done[grp];
                    const uint32_t fb = tc::smem_u32(&full_bar[st]);
                    if (!lp) {
                        // only the peer issued this fill: the leader's arrivals, expecting what came
                        tc::mbar_arrive_expect_tx(fb, (pp ? b : 0u) + (ps ? (uint32_t)kSignalBytes : 0u));
                        if (QW) tc::mbar_arrive(fb);
                    } else {
                        const uint32_t missing =
                            (PAIR && !pp ? b : 0u) + (QW && PAIR && main && !ps ? (uint32_t)kSignalBytes : 0u);
                        if (missing) tc::mbar_complete_tx(fb, missing);
                        if (QW && main && !lc) tc::mbar_arrive(fb);
                    }
                    tc::mbar_wait(tc::smem_u32(&full_bar[st]), (uint32_t)(f / kStages) & 1u);
                }
            }
        } else if (warp == 1 && lane == 0 && rank == 0) {
            // completes when every MMA this thread issued has completed
            if constexpr (PAIR) tc::mma_commit_pair(tc::smem_u32(drain_bar), 0x1);
            else tc::mma_commit(tc::smem_u32(drain_bar));
            tc::mbar_wait(tc::smem_u32(drain_bar), 0);
        }
        tc::fence_before_sync();
        __syncthreads();
        if constexpr (PAIR) tc::cluster_sync();
    }
    if (warp == 1) {
        tc::fence_after_sync();
        if constexpr (PAIR) tc::tmem_dealloc_pair(tmem_base, kTmemCols);
        else tc::tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

CUtensorMapSwizzle swizzle_for_bytes(int inner_bytes) {
    return inner_bytes >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                              : (inner_bytes >= 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

bool encode(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
            const uint32_t* box, CUtensorMapSwizzle sw,
            CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t gd[3], gs[2];
    cuuint32_t bx[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
    }
    for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
    return fn(m, dt, rank, const_cast<void*>(base), gd, gs, bx, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
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

// One CTA per SM (grid = min(#SMs, tiles)); SM pairs: as many 2-CTA clusters as can be
// resident at once (so that no pair waits for another to finish), at most one per tile.
template <int EPI, bool B_MN, int BN, bool PAIR, int QB = 0, int CG = 0>
cudaError_t launch_tc(const TcParams& P, int64_t max_tiles, size_t smem, cudaStream_t s) {
    auto k = grouped_gemm_tc_kernel<EPI, B_MN, BN, PAIR, QB, CG>;
    constexpr int kThr = threads_of(CG);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if constexpr (!PAIR) {
        const int grid = (int)std::min<int64_t>(sm_count(), max_tiles);
        return launch_pdl(k, dim3(grid), dim3(kThr), smem, s, P);
    } else {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.blockDim = dim3(kThr, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3((unsigned)(sm_count() & ~1), 1, 1);
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, k, &cfg);
        if (e != cudaSuccess) return e;
        if (clusters < 1) return cudaErrorNotSupported;     // caller falls back to single-CTA tiles
        const int64_t pairs = std::min<int64_t>(clusters, max_tiles);
        cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see launch_pdl
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, k, P);
    }
}

// The layer's four expert GEMMs with quantised weights (QB-bit codes, CG converter groups)
template <int QB, int CG>
cudaError_t launch_quant(const TcParams& P, const GroupedGemm& g, int64_t max_tiles, size_t offs_bytes,
                         cudaStream_t s) {
    const size_t smem = Geo<256, true, QB>::kSmem + offs_bytes;
    switch (g.epi) {
        case EPI_SWIGLU: return launch_tc<EPI_SWIGLU, true, 256, true, QB, CG>(P, max_tiles, smem, s);
        case EPI_BF16:
            return g.b_mn_major ? launch_tc<EPI_BF16, true, 256, true, QB, CG>(P, max_tiles, smem, s)
                                : launch_tc<EPI_BF16, false, 256, true, QB, CG>(P, max_tiles, smem, s);
        default: return launch_tc<EPI_DSWIGLU, false, 256, true, QB, CG>(P, max_tiles, smem, s);
    }
}

// SM pairs halve the B bytes each SM pulls through L2 per flop but pad every expert
// to 256-row tiles; they pay off when experts average at least MOE_PAIR_MIN_ROWS rows.
#ifndef MOE_PAIR_MIN_ROWS
#define MOE_PAIR_MIN_ROWS 384
#endif
bool use_sm_pairs(const GroupedGemm& g) { return g.N >= (int64_t)MOE_PAIR_MIN_ROWS * g.E; }

}  // namespace

namespace {

cudaError_t launch_impl(const GroupedGemm& g, bool allow_pairs, cudaStream_t s) {
    if (g.K % BK != 0) return cudaErrorInvalidValue;
    const bool proj = g.epi == EPI_PROJ;
    const int BN = proj ? g.Ncols : 256;
    if (proj && (g.b_mn_major || g.A2 != nullptr || (BN != 16 && BN != 32 && BN != 64))) return cudaErrorInvalidValue;
    if (!proj && g.Ncols % 64 != 0) return cudaErrorInvalidValue;
    if (g.epi == EPI_SWIGLU && !g.b_mn_major) return cudaErrorInvalidValue;   // gate/up pairing needs MN-major B
    TcParams P;
    memset(&P, 0, sizeof(P));
    P.g = g;
    P.num_kb = g.K / BK;
    P.wait_ns = tc::kWaitTimeoutNs;
    const bool paired = g.epi == EPI_SWIGLU;
    const int qb = g.b_quant;                       // bits per code of a quantised B (0: bf16)
    if (qb != 0 && qb != 8 && qb != 4) return cudaErrorInvalidValue;
    if (qb != 0 && g.b_scale == nullptr) return cudaErrorInvalidValue;
    // quantised weights always run on SM pairs: each CTA dequantises half of the B tile
    const bool pair = allow_pairs && !proj && (qb != 0 || use_sm_pairs(g));
    if (qb != 0 && (proj || g.ldb % 64 != 0)) return cudaErrorInvalidValue;
    if (qb == 4) memcpy(P.nf4, nf4_table().v, sizeof(P.nf4));
    // kernels exist for the layer's four expert GEMMs (below) and the projections
    if (!proj && g.epi != EPI_SWIGLU && g.epi != EPI_BF16 && g.epi != EPI_DSWIGLU) return cudaErrorInvalidValue;
    if (g.epi == EPI_DSWIGLU && g.b_mn_major) return cudaErrorInvalidValue;   // built for a K-major B only
    P.n_tiles = proj ? 1 : (paired ? (g.Ncols + 127) / 128 : (g.Ncols + 255) / 256);
    // A: [N, K]
    {
        const uint64_t dims[2] = {(uint64_t)g.K, (uint64_t)g.N};
        const uint64_t st[1] = {(uint64_t)g.K * 2};
        const uint32_t box[2] = {BK, BM};
        if (!encode(&P.tm_a, g.A, 2, dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
        const uint32_t box64[2] = {BK, BM / 2};      // half tiles of SM pairs
        if (pair && !encode(&P.tm_a64, g.A, 2, dims, st, box64, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    }
    // B: expert stack
    {
        const uint64_t rows = (uint64_t)(g.b_expert_stride / g.ldb);
        const uint64_t dims[3] = {(uint64_t)g.ldb, rows, (uint64_t)g.E};
        const uint64_t st[2] = {(uint64_t)g.ldb * 2, (uint64_t)g.b_expert_stride * 2};
        const uint32_t box_mn[3] = {64, BK, 1};
        const uint32_t box_k[3] = {BK, (uint32_t)(pair ? BN / 2 : BN), 1};
        if (qb != 0) {
            // codes landed unswizzled in the staging slot, addressed as bytes: e4m3 one per
            // byte, NF4 two per byte (a 64-element row of a box is 32 bytes)
            const uint64_t dims_q[3] = {(uint64_t)g.ldb * qb / 8, rows, (uint64_t)g.E};
            const uint64_t st_q[2] = {(uint64_t)g.ldb * qb / 8, (uint64_t)g.b_expert_stride * qb / 8};
            const uint32_t box_mn_q[3] = {(uint32_t)(64 * qb / 8), BK, 1};
            const uint32_t box_k_q[3] = {(uint32_t)(BK * qb / 8), (uint32_t)(BN / 2), 1};
            if (!encode(&P.tm_b, g.B, 3, dims_q, st_q, g.b_mn_major ? box_mn_q : box_k_q, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_DATA_TYPE_UINT8))
                return cudaErrorInvalidValue;
            if (qb == 4) {
                // block scales [E][ldb / 64][rows] float32: a stage takes 64 k rows of one column
                // block (MN-major B) or 128 n rows of one k block (K-major B)
                const uint64_t nblk = (uint64_t)g.ldb / 64;
                const uint64_t dims_s[3] = {rows, nblk, (uint64_t)g.E};
                const uint64_t st_s[2] = {rows * 4, rows * nblk * 4};
                const uint32_t box_s[3] = {g.b_mn_major ? 64u : (uint32_t)(BN / 2), 1, 1};
                if (!encode(&P.tm_bs, g.b_scale, 3, dims_s, st_s, box_s, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
                    return cudaErrorInvalidValue;
            }
        } else if (!encode(&P.tm_b, g.B, 3, dims, st, g.b_mn_major ? box_mn : box_k, CU_TENSOR_MAP_SWIZZLE_128B)) {
            return cudaErrorInvalidValue;
        }
    }
    if (g.A2 != nullptr && g.r > 0) {
        const int rp = g.rp;
        P.lora_k16 = rp / 16;
        const uint64_t dims[2] = {(uint64_t)rp, (uint64_t)g.N};
        const uint64_t st[1] = {(uint64_t)rp * 2};
        const uint32_t box[2] = {(uint32_t)rp, BM};
        if (!encode(&P.tm_a2, g.A2, 2, dims, st, box, swizzle_for_bytes(rp * 2))) return cudaErrorInvalidValue;
        const uint32_t box64[2] = {(uint32_t)rp, BM / 2};
        if (pair && !encode(&P.tm_a2_64, g.A2, 2, dims, st, box64, swizzle_for_bytes(rp * 2)))
            return cudaErrorInvalidValue;
        P.a2_bytes = BM * rp * 2;
        P.a2_sbo = 8 * rp * 2;
        P.a2_swz = rp >= 64 ? tc::kSw128 : (rp >= 32 ? tc::kSw64 : tc::kSw32);
        const uint64_t dims2[3] = {(uint64_t)g.ldb2, (uint64_t)g.r, (uint64_t)g.E};
        const uint64_t st2[2] = {(uint64_t)g.ldb2 * 2, (uint64_t)g.b2_expert_stride * 2};
        const uint32_t box2[3] = {64, (uint32_t)rp, 1};
        if (!encode(&P.tm_b2, g.B2, 3, dims2, st2, box2, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
        P.b2_box_bytes = 64 * rp * 2;
    }
    const int64_t tm = pair ? 2 * BM : BM;
    const int64_t max_tiles = ((g.N + tm - 1) / tm + g.E) * (int64_t)P.n_tiles;
    if (!pair) {
        // diagnostics: a single-CTA launch the caller chose to fail (moe_diag_force_timeout)
        const DiagWait dw = diag_next_single_cta_launch();
        if (dw.stall) {
            P.stall = 1;
            P.wait_ns = dw.limit_ns;
        }
    }
    const size_t offs_bytes = (size_t)2 * (g.E + 1) * sizeof(int32_t);
    const bool mn = g.b_mn_major;
    if (proj) {
        switch (BN) {
            case 16: return launch_tc<EPI_PROJ, false, 16, false>(P, max_tiles, Geo<16>::kSmem + offs_bytes, s);
            case 32: return launch_tc<EPI_PROJ, false, 32, false>(P, max_tiles, Geo<32>::kSmem + offs_bytes, s);
            default: return launch_tc<EPI_PROJ, false, 64, false>(P, max_tiles, Geo<64>::kSmem + offs_bytes, s);
        }
    }
    // The layer's expert GEMMs: gate_up forward (SwiGLU, MN-major B), down forward (bf16,
    // MN-major B), down backward (SwiGLU backward, K-major B: W_d read transposed) and
    // gate_up backward (bf16, K-major B: W_gu read transposed).
    if (qb != 0) {
        if (!pair) return cudaErrorNotSupported;   // quantised weights run on SM pairs only
        // three converter groups (and a 4-warp epilogue) for long k loops, or for half tiles
        // (experts of under 256 rows on average) with k >= 2048; two groups (8 epilogue warps)
        // where each tile's epilogue must hide behind a short k loop
        const bool three = g.K >= 2560 || (g.N < 256 * (int64_t)g.E && g.K >= 2048);
        if (qb == 8) return three ? launch_quant<8, 3>(P, g, max_tiles, offs_bytes, s)
                                  : launch_quant<8, 2>(P, g, max_tiles, offs_bytes, s);
        return three ? launch_quant<4, 3>(P, g, max_tiles, offs_bytes, s)
                     : launch_quant<4, 2>(P, g, max_tiles, offs_bytes, s);
    }
    if (pair) {
        const size_t smem = Geo<256, true>::kSmem + offs_bytes;
        switch (g.epi) {
            case EPI_SWIGLU: return launch_tc<EPI_SWIGLU, true, 256, true>(P, max_tiles, smem, s);
            case EPI_BF16:
                return mn ? launch_tc<EPI_BF16, true, 256, true>(P, max_tiles, smem, s)
                          : launch_tc<EPI_BF16, false, 256, true>(P, max_tiles, smem, s);
            default: return launch_tc<EPI_DSWIGLU, false, 256, true>(P, max_tiles, smem, s);
        }
    }
    const size_t smem = Geo<256>::kSmem + offs_bytes;
    switch (g.epi) {
        case EPI_SWIGLU: return launch_tc<EPI_SWIGLU, true, 256, false>(P, max_tiles, smem, s);
        case EPI_BF16:
            return mn ? launch_tc<EPI_BF16, true, 256, false>(P, max_tiles, smem, s)
                      : launch_tc<EPI_BF16, false, 256, false>(P, max_tiles, smem, s);
        default: return launch_tc<EPI_DSWIGLU, false, 256, false>(P, max_tiles, smem, s);
    }
}

}  // namespace

cudaError_t launch_grouped_gemm(const GroupedGemm& g, cudaStream_t s) {
    if (g.N == 0) return cudaSuccess;
    const cudaError_t e = launch_impl(g, true, s);
    // no resident 2-CTA cluster fits on this device: single-CTA tiles
    if (e == cudaErrorNotSupported) return launch_impl(g, false, s);
    return e;
}

}  // namespace moe
