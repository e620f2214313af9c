// C ABI of the MoE-LoRA expert layer: argument checks, buffer carving and the
// launch sequences of route / forward / backward.  Nothing here waits on the
// device or copies to the host.
#include "common.cuh"
#include "kernels.h"

#include <atomic>
#include <mutex>
#include <string.h>
#include <vector>

#include "tc_ptx.cuh"

using namespace moe;

namespace {

// ---- diagnostics: a chosen single-CTA tensor-core launch fails on purpose
struct ForcedTimeout {
    std::atomic<int64_t> target{-1};      // index of the launch to fail among those counted, -1: none
    std::atomic<int64_t> seen{0};         // single-CTA tensor-core launches counted since arming
    std::atomic<uint64_t> limit_ns{tc::kWaitTimeoutNs};
};

ForcedTimeout& forced() {
    static ForcedTimeout f;
    return f;
}

// ---- diagnostics: per-kernel CUDA-event timing and a launch counter
struct TimedLaunch {
    const char* name;
    cudaEvent_t start, stop;
};

struct Timing {
    std::mutex mu;
    bool on = false;
    std::vector<TimedLaunch> pool;   // events are created once and reused
    size_t used = 0;
    unsigned long long launches = 0;
};

Timing& timing() {
    static Timing t;
    return t;
}

// Run one kernel-launching expression, bracketed by events when timing is on.
template <typename F>
cudaError_t timed(const char* name, cudaStream_t s, F&& f, int n_ops = 1) {
    Timing& t = timing();
    // the event handles are copied out under the lock: another thread's push_back may move
    // the pool's elements
    cudaEvent_t ev_start = nullptr, ev_stop = nullptr;
    {
        std::lock_guard<std::mutex> g(t.mu);
        t.launches += n_ops;
        if (t.on) {
            if (t.used == t.pool.size()) {
                TimedLaunch tl{name, nullptr, nullptr};
                if (cudaEventCreate(&tl.start) != cudaSuccess) return cudaErrorMemoryAllocation;
                if (cudaEventCreate(&tl.stop) != cudaSuccess) {
                    cudaEventDestroy(tl.start);
                    return cudaErrorMemoryAllocation;
                }
                t.pool.push_back(tl);
            }
            TimedLaunch& slot = t.pool[t.used++];
            slot.name = name;
            ev_start = slot.start;
            ev_stop = slot.stop;
        }
    }
    if (ev_start) cudaEventRecord(ev_start, s);
    cudaError_t e = f();
    if (ev_stop) cudaEventRecord(ev_stop, s);
    return e;
}

constexpr size_t kAlign = 256;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// activation rows (x, y, dy, dx and the saved / workspace buffers) are moved with 32-byte
// accesses, one full L2 sector per thread
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

moe_status check_dims(const moe_dims* d) {
    if (d == nullptr) return MOE_ERR_NULL_ARG;
    if (d->T < 0 || d->k < 1 || d->E < 1 || d->k > d->E || d->E > 1024) return MOE_ERR_BAD_DIMS;
    if (d->H <= 0 || d->I <= 0 || d->H % 64 != 0 || d->I % 64 != 0) return MOE_ERR_BAD_DIMS;
    if (d->r < 1 || d->r > 64) return MOE_ERR_BAD_DIMS;
    if (d->T * (int64_t)d->k >= (int64_t(1) << 31)) return MOE_ERR_BAD_DIMS;
    return MOE_OK;
}

// perm / inv_perm / w_sorted have N = T*k entries and may be NULL when N == 0.
moe_status check_routing(const moe_routing* rt, int64_t N) {
    if (rt == nullptr || rt->counts == nullptr || rt->offsets == nullptr || rt->tile_offsets == nullptr)
        return MOE_ERR_NULL_ARG;
    if (N > 0 && (rt->perm == nullptr || rt->inv_perm == nullptr || rt->w_sorted == nullptr))
        return MOE_ERR_NULL_ARG;
    if (!aligned16(rt->perm) || !aligned16(rt->inv_perm) || !aligned16(rt->w_sorted))
        return MOE_ERR_MISALIGNED;
    return MOE_OK;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

struct SavedLayout {
    size_t x_perm, gu, h, xa, ha, o, total;
    int rp;
};

SavedLayout saved_layout(const moe_dims* d) {
    const size_t N = (size_t)d->T * d->k;
    SavedLayout L;
    L.rp = lora_rp(d->r);
    size_t o = 0;
    L.x_perm = o; o = align_up(o + N * d->H * 2, kAlign);
    L.gu = o;     o = align_up(o + N * 2 * d->I * 2, kAlign);
    L.h = o;      o = align_up(o + N * d->I * 2, kAlign);
    L.xa = o;     o = align_up(o + N * L.rp * 2, kAlign);
    L.ha = o;     o = align_up(o + N * L.rp * 2, kAlign);
    L.o = o;      o = align_up(o + N * d->H * 2, kAlign);
    L.total = o;
    return L;
}

// The forward needs no workspace (every intermediate is kept in `saved`).
struct FwdWs {
    size_t total;
};

FwdWs fwd_ws(const moe_dims*) { return FwdWs{0}; }

struct BwdWs {
    size_t d_o, g_s, dgu, gg_s, dx_perm, total;
};

BwdWs bwd_ws(const moe_dims* d) {
    const size_t N = (size_t)d->T * d->k;
    const int rp = lora_rp(d->r);
    BwdWs W;
    size_t o = 0;
    W.d_o = o;     o = align_up(o + N * d->H * 2, kAlign);
    W.g_s = o;     o = align_up(o + N * rp * 2, kAlign);
    W.dgu = o;     o = align_up(o + N * 2 * d->I * 2, kAlign);
    W.gg_s = o;    o = align_up(o + N * rp * 2, kAlign);
    W.dx_perm = o; o = align_up(o + N * d->H * 2, kAlign);
    W.total = o;
    return W;
}

// Rank-r projection P = s * In Wt[e]^T on the tensor cores (tile width RP).
cudaError_t project(const void* In, int K, const void* Wt, int r, int rp, float scale, const moe_routing* rt,
                    int E, int64_t N, void* P, int32_t* dev_status, cudaStream_t s) {
    GroupedGemm g{};
    g.N = N; g.E = E; g.K = K; g.Ncols = rp;
    g.A = In; g.B = Wt; g.b_mn_major = false; g.ldb = K; g.b_expert_stride = (int64_t)r * K;
    g.offsets = rt->offsets; g.tile_offsets = rt->tile_offsets;
    g.out0 = P; g.scale = scale; g.epi = EPI_PROJ; g.dev_status = dev_status;
    return launch_grouped_gemm(g, s);
}

#define MOE_TRY(expr)                                  \
    do {                                               \
        cudaError_t _e = (expr);                       \
        if (_e != cudaSuccess) return MOE_ERR_CUDA;    \
    } while (0)

}  // namespace

DiagWait moe::diag_next_single_cta_launch() {
    ForcedTimeout& f = forced();
    const int64_t target = f.target.load();
    if (target >= 0 && f.seen.fetch_add(1) == target) {
        int64_t expect = target;
        if (f.target.compare_exchange_strong(expect, -1)) return DiagWait{f.limit_ns.load(), true};
    }
    return DiagWait{tc::kWaitTimeoutNs, false};
}

extern "C" {

int32_t moe_abi_version(void) { return 7; }

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_NULL_ARG: return "a required pointer is NULL";
        case MOE_ERR_BAD_DIMS: return "sizes outside the supported range";
        case MOE_ERR_MISALIGNED: return "a pointer is not 16-byte aligned (activation buffers: 32-byte)";
        case MOE_ERR_WORKSPACE: return "workspace or saved buffer too small";
        case MOE_ERR_CUDA: return "a CUDA call failed";
        case MOE_ERR_UNSUPPORTED: return "unsupported device or driver";
        default: return "unknown status";
    }
}

moe_status moe_route_workspace_size(int64_t T, int32_t k, int32_t E, size_t* bytes) {
    if (bytes == nullptr) return MOE_ERR_NULL_ARG;
    if (T < 0 || k < 1 || E < 1 || k > E || E > 1024 || T * (int64_t)k >= (int64_t(1) << 31))
        return MOE_ERR_BAD_DIMS;
    *bytes = route_workspace_bytes(T * (int64_t)k, E);
    return MOE_OK;
}

moe_status moe_route(const void* topk_idx, int32_t idx_bytes, const float* topk_w, int64_t T, int32_t k,
                     int32_t E, const moe_routing* out, void* workspace, size_t workspace_bytes,
                     int32_t* dev_status, void* stream) {
    size_t need = 0;
    moe_status st = moe_route_workspace_size(T, k, E, &need);
    if (st != MOE_OK) return st;
    if (idx_bytes != 4 && idx_bytes != 8) return MOE_ERR_BAD_DIMS;
    if ((T > 0 && (topk_idx == nullptr || topk_w == nullptr)) || workspace == nullptr || dev_status == nullptr)
        return MOE_ERR_NULL_ARG;
    if ((st = check_routing(out, T * (int64_t)k)) != MOE_OK) return st;
    if (!aligned16(workspace) || (T > 0 && (!aligned16(topk_idx) || !aligned16(topk_w))))
        return MOE_ERR_MISALIGNED;
    if (workspace_bytes < need) return MOE_ERR_WORKSPACE;
    return cuda_status(timed("route", (cudaStream_t)stream, [&] {
        return launch_route(topk_idx, idx_bytes, topk_w, T * (int64_t)k, E, *out, workspace, dev_status,
                            (cudaStream_t)stream);
    }, T > 0 ? 3 : 2));
}

moe_status moe_route_static(const void* topk_idx, int32_t idx_bytes, const float* topk_w, int64_t T, int32_t k,
                            int32_t E, const moe_routing* out, int32_t* dev_status, void* stream) {
    size_t need = 0;
    moe_status st = moe_route_workspace_size(T, k, E, &need);
    if (st != MOE_OK) return st;
    if (need > MOE_ROUTE_STATIC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
    if (idx_bytes != 4 && idx_bytes != 8) return MOE_ERR_BAD_DIMS;
    if ((T > 0 && (topk_idx == nullptr || topk_w == nullptr)) || dev_status == nullptr) return MOE_ERR_NULL_ARG;
    if ((st = check_routing(out, T * (int64_t)k)) != MOE_OK) return st;
    if (T > 0 && (!aligned16(topk_idx) || !aligned16(topk_w))) return MOE_ERR_MISALIGNED;
    void* scratch = nullptr;
    if (route_static_scratch(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_status(timed("route", (cudaStream_t)stream, [&] {
        return launch_route(topk_idx, idx_bytes, topk_w, T * (int64_t)k, E, *out, scratch, dev_status,
                            (cudaStream_t)stream);
    }, T > 0 ? 3 : 2));
}

moe_status moe_lora_fwd_sizes(const moe_dims* d, size_t* saved_bytes, size_t* workspace_bytes) {
    moe_status st = check_dims(d);
    if (st != MOE_OK) return st;
    if (saved_bytes == nullptr || workspace_bytes == nullptr) return MOE_ERR_NULL_ARG;
    *saved_bytes = saved_layout(d).total;
    *workspace_bytes = fwd_ws(d).total;
    return MOE_OK;
}

moe_status moe_lora_saved_layout(const moe_dims* d, size_t offsets[6], int32_t* rp) {
    moe_status st = check_dims(d);
    if (st != MOE_OK) return st;
    if (offsets == nullptr || rp == nullptr) return MOE_ERR_NULL_ARG;
    const SavedLayout L = saved_layout(d);
    offsets[0] = L.x_perm; offsets[1] = L.gu; offsets[2] = L.h; offsets[3] = L.xa; offsets[4] = L.ha;
    offsets[5] = L.o;
    *rp = L.rp;
    return MOE_OK;
}

moe_status moe_lora_saved_regather(const moe_dims* d, const moe_routing* rt, const uint16_t* x, void* saved,
                                   size_t saved_bytes, void* stream) {
    moe_status st = check_dims(d);
    if (st != MOE_OK) return st;
    const int64_t N = d->T * (int64_t)d->k;
    if ((st = check_routing(rt, N)) != MOE_OK) return st;
    if (N > 0 && (x == nullptr || saved == nullptr)) return MOE_ERR_NULL_ARG;
    if (!aligned32(x) || !aligned32(saved)) return MOE_ERR_MISALIGNED;
    const SavedLayout L = saved_layout(d);
    if (saved_bytes < L.total) return MOE_ERR_WORKSPACE;
    if (N == 0) return MOE_OK;
    cudaStream_t s = (cudaStream_t)stream;
    void* x_perm = static_cast<uint8_t*>(saved) + L.x_perm;
    MOE_TRY(timed("gather_x", s, [&] {
        return launch_gather_rows(x, d->H, rt->perm, nullptr, N, d->k, x_perm, nullptr, nullptr, nullptr, s);
    }));
    return MOE_OK;
}

moe_status moe_lora_saved_rebuild_h(const moe_dims* d, void* saved, size_t saved_bytes, void* stream) {
    moe_status st = check_dims(d);
    if (st != MOE_OK) return st;
    const int64_t N = d->T * (int64_t)d->k;
    if (N > 0 && saved == nullptr) return MOE_ERR_NULL_ARG;
    if (!aligned32(saved)) return MOE_ERR_MISALIGNED;
    const SavedLayout L = saved_layout(d);
    if (saved_bytes < L.total) return MOE_ERR_WORKSPACE;
    if (N == 0) return MOE_OK;
    cudaStream_t s = (cudaStream_t)stream;
    uint8_t* sv = static_cast<uint8_t*>(saved);
    MOE_TRY(timed("rebuild_h", s, [&] { return launch_swiglu_rows(sv + L.gu, d->I, N, sv + L.h, s); }));
    return MOE_OK;
}

moe_status moe_lora_bwd_workspace_size(const moe_dims* d, size_t* bytes) {
    moe_status st = check_dims(d);
    if (st != MOE_OK) return st;
    if (bytes == nullptr) return MOE_ERR_NULL_ARG;
    *bytes = bwd_ws(d).total;
    return MOE_OK;
}

// Forward / backward launch sequences.  qbits 8: W_gu / W_d hold e4m3 codes with per-column
// power-of-two scales s_gu / s_d; qbits 4: NF4 codes with one absmax per 64 elements of a row;
// both dequantised inside the GEMM pipeline.  qbits 0: bf16 weights (s_gu, s_d unused).
static moe_status fwd_impl(const moe_dims* d, const moe_routing* rt, const uint16_t* x, const void* W_gu,
                           const float* s_gu, const uint16_t* A_gu, const uint16_t* B_gu, const void* W_d,
                           const float* s_d, const uint16_t* A_d, const uint16_t* B_d, uint16_t* y, void* saved,
                           size_t saved_bytes, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           void* stream, int qbits = 0, bool h_from_gu = false) {
    if (!aligned16(s_gu) || !aligned16(s_d)) return MOE_ERR_MISALIGNED;
    moe_status st = check_dims(d);
    if (st != MOE_OK) return st;
    const int64_t Nr = d->T * (int64_t)d->k;
    if ((st = check_routing(rt, Nr)) != MOE_OK) return st;
    // token-sized buffers may be NULL when T == 0; the forward workspace is unused (size 0)
    const void* tok[] = {x, y, saved};
    const void* always[] = {W_gu, A_gu, B_gu, W_d, A_d, B_d, dev_status};
    for (const void* p : always) if (p == nullptr) return MOE_ERR_NULL_ARG;
    if (Nr > 0) for (const void* p : tok) if (p == nullptr) return MOE_ERR_NULL_ARG;
    for (const void* p : always) if (!aligned16(p)) return MOE_ERR_MISALIGNED;
    for (const void* p : tok) if (!aligned32(p)) return MOE_ERR_MISALIGNED;
    if (!aligned32(workspace)) return MOE_ERR_MISALIGNED;
    const SavedLayout L = saved_layout(d);
    const FwdWs W = fwd_ws(d);
    if (saved_bytes < L.total || workspace_bytes < W.total) return MOE_ERR_WORKSPACE;
    const int64_t N = d->T * (int64_t)d->k;
    if (N == 0) return MOE_OK;
    cudaStream_t s = (cudaStream_t)stream;
    char* sv = (char*)saved;
    void* x_perm = sv + L.x_perm;
    void* GU = sv + L.gu;
    void* h = sv + L.h;
    void* XA = sv + L.xa;
    void* HA = sv + L.ha;
    void* O = sv + L.o;
    const int H = d->H, I = d->I, E = d->E, r = d->r;

    MOE_TRY(timed("gather_x", s, [&] { return launch_gather_rows(x, H, rt->perm, nullptr, N, d->k, x_perm, nullptr, nullptr, dev_status, s); }));
    MOE_TRY(timed("proj_xa", s, [&] { return project(x_perm, H, A_gu, r, L.rp, d->scale, rt, E, N, XA, dev_status, s); }));

    GroupedGemm g{};
    g.N = N; g.E = E; g.offsets = rt->offsets; g.tile_offsets = rt->tile_offsets; g.dev_status = dev_status;
    // gate_up: GU = x_perm W_gu[e] + XA_s B_gu[e]; h = silu(g) * u
    g.K = H; g.Ncols = I; g.A = x_perm;
    g.B = W_gu; g.b_quant = qbits; g.b_scale = s_gu; g.b_mn_major = true; g.ldb = 2 * I; g.b_expert_stride = (int64_t)H * 2 * I;
    g.A2 = XA; g.rp = L.rp; g.r = r; g.B2 = B_gu; g.ldb2 = 2 * I; g.b2_expert_stride = (int64_t)r * 2 * I;
    g.out0 = GU; g.out1 = h; g.epi = EPI_SWIGLU; g.h_from_gu = h_from_gu ? 1 : 0;
    MOE_TRY(timed("gemm_gate_up_fwd", s, [&] { return launch_grouped_gemm(g, s); }));

    MOE_TRY(timed("proj_ha", s, [&] { return project(h, I, A_d, r, L.rp, d->scale, rt, E, N, HA, dev_status, s); }));
    // down: O = h W_d[e] + HA_s B_d[e]  (unweighted, kept for the routing-weight gradient)
    GroupedGemm g2{};
    g2.N = N; g2.E = E; g2.offsets = rt->offsets; g2.tile_offsets = rt->tile_offsets; g2.dev_status = dev_status;
    g2.K = I; g2.Ncols = H; g2.A = h;
    g2.B = W_d; g2.b_quant = qbits; g2.b_scale = s_d; g2.b_mn_major = true; g2.ldb = H; g2.b_expert_stride = (int64_t)I * H;
    g2.A2 = HA; g2.rp = L.rp; g2.r = r; g2.B2 = B_d; g2.ldb2 = H; g2.b2_expert_stride = (int64_t)r * H;
    g2.out0 = O; g2.ldo = H; g2.epi = EPI_BF16;
    MOE_TRY(timed("gemm_down_fwd", s, [&] { return launch_grouped_gemm(g2, s); }));

    MOE_TRY(timed("combine_y", s, [&] { return launch_combine(O, rt->w_sorted, rt->inv_perm, d->T, d->k, H, y, dev_status, s); }));
    return MOE_OK;
}

static moe_status bwd_impl(const moe_dims* d, const moe_routing* rt, const uint16_t* dy, const void* W_gu,
                           const float* s_gu, const uint16_t* A_gu, const uint16_t* B_gu, const void* W_d,
                           const float* s_d, const uint16_t* A_d, const uint16_t* B_d, const void* saved,
                           size_t saved_bytes, uint16_t* dx, uint16_t* dA_gu, uint16_t* dB_gu, uint16_t* dA_d,
                           uint16_t* dB_d, float* d_topk_w, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, void* stream, int qbits = 0) {
    if (!aligned16(s_gu) || !aligned16(s_d)) return MOE_ERR_MISALIGNED;
    moe_status st = check_dims(d);
    if (st != MOE_OK) return st;
    const int64_t Nr = d->T * (int64_t)d->k;
    if ((st = check_routing(rt, Nr)) != MOE_OK) return st;
    // token-sized buffers may be NULL when T == 0
    const void* tok[] = {dy, saved, dx, workspace};
    const void* always[] = {W_gu, A_gu, B_gu, W_d, A_d, B_d, dA_gu, dB_gu, dA_d, dB_d, dev_status};
    for (const void* p : always) if (p == nullptr) return MOE_ERR_NULL_ARG;
    if (Nr > 0) for (const void* p : tok) if (p == nullptr) return MOE_ERR_NULL_ARG;
    for (const void* p : always) if (!aligned16(p)) return MOE_ERR_MISALIGNED;
    for (const void* p : tok) if (!aligned32(p)) return MOE_ERR_MISALIGNED;
    if (!aligned16(d_topk_w)) return MOE_ERR_MISALIGNED;
    const SavedLayout L = saved_layout(d);
    const BwdWs W = bwd_ws(d);
    if (saved_bytes < L.total || workspace_bytes < W.total) return MOE_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t N = d->T * (int64_t)d->k;
    const int H = d->H, I = d->I, E = d->E, r = d->r;
    if (N == 0) {
        MOE_TRY(cudaMemsetAsync(dA_gu, 0, (size_t)E * r * H * 2, s));
        MOE_TRY(cudaMemsetAsync(dB_gu, 0, (size_t)E * r * 2 * I * 2, s));
        MOE_TRY(cudaMemsetAsync(dA_d, 0, (size_t)E * r * I * 2, s));
        MOE_TRY(cudaMemsetAsync(dB_d, 0, (size_t)E * r * H * 2, s));
        return MOE_OK;
    }
    const char* sv = (const char*)saved;
    const void* x_perm = sv + L.x_perm;
    const void* GU = sv + L.gu;
    const void* h = sv + L.h;
    const void* XA = sv + L.xa;
    const void* HA = sv + L.ha;
    const void* Os = sv + L.o;
    char* ws = (char*)workspace;
    void* dO = ws + W.d_o;
    void* G = ws + W.g_s;
    void* dGU = ws + W.dgu;
    void* Gg = ws + W.gg_s;
    void* dXp = ws + W.dx_perm;

    // dO = w * dy[token]  (and d_topk_w[slot] = <dy[token], O[p]> when requested)
    MOE_TRY(timed("gather_dy", s, [&] { return launch_gather_rows(dy, H, rt->perm, rt->w_sorted, N, d->k, dO, Os, d_topk_w, dev_status, s); }));
    // G_s = s * dO B_d^T
    MOE_TRY(timed("proj_g", s, [&] { return project(dO, H, B_d, r, L.rp, d->scale, rt, E, N, G, dev_status, s); }));
    // dh = dO W_d[e]^T + G_s A_d[e]  ->  dGU = SwiGLU'(GU) dh
    GroupedGemm g{};
    g.N = N; g.E = E; g.offsets = rt->offsets; g.tile_offsets = rt->tile_offsets; g.dev_status = dev_status;
    g.K = H; g.Ncols = I; g.A = dO;
    g.B = W_d; g.b_quant = qbits; g.b_scale = s_d; g.b_mn_major = false; g.ldb = H; g.b_expert_stride = (int64_t)I * H;
    g.A2 = G; g.rp = L.rp; g.r = r; g.B2 = A_d; g.ldb2 = I; g.b2_expert_stride = (int64_t)r * I;
    g.gu_in = GU; g.out0 = dGU; g.epi = EPI_DSWIGLU;
    MOE_TRY(timed("gemm_down_bwd", s, [&] { return launch_grouped_gemm(g, s); }));
    // dA_d = G_s^T h ; dB_d = HA_s^T dO
    {
        const WgradProblem wp[2] = {{G, h, I, dA_d}, {HA, dO, H, dB_d}};
        MOE_TRY(timed("wgrad_down", s, [&] { return launch_lora_wgrad_tc(wp, 2, L.rp, r, rt->offsets, E, N, dev_status, s); }));
    }
    // Gg_s = s * dGU B_gu^T
    MOE_TRY(timed("proj_gg", s, [&] { return project(dGU, 2 * I, B_gu, r, L.rp, d->scale, rt, E, N, Gg, dev_status, s); }));
    // dX_perm = dGU W_gu[e]^T + Gg_s A_gu[e], one bf16 row per routed slot (like the forward's
    // O rows); the combine sums a token's k slots in fp32
    GroupedGemm g2{};
    g2.N = N; g2.E = E; g2.offsets = rt->offsets; g2.tile_offsets = rt->tile_offsets; g2.dev_status = dev_status;
    g2.K = 2 * I; g2.Ncols = H; g2.A = dGU;
    g2.B = W_gu; g2.b_quant = qbits; g2.b_scale = s_gu; g2.b_mn_major = false; g2.ldb = 2 * I; g2.b_expert_stride = (int64_t)H * 2 * I;
    g2.A2 = Gg; g2.rp = L.rp; g2.r = r; g2.B2 = A_gu; g2.ldb2 = H; g2.b2_expert_stride = (int64_t)r * H;
    g2.out0 = dXp; g2.ldo = H; g2.epi = EPI_BF16;
    MOE_TRY(timed("gemm_gate_up_bwd", s, [&] { return launch_grouped_gemm(g2, s); }));
    MOE_TRY(timed("combine_dx", s, [&] { return launch_combine(dXp, nullptr, rt->inv_perm, d->T, d->k, H, dx, dev_status, s); }));
    // dA_gu = Gg_s^T x_perm ; dB_gu = XA_s^T dGU
    {
        const WgradProblem wp[2] = {{Gg, x_perm, H, dA_gu}, {XA, dGU, 2 * I, dB_gu}};
        MOE_TRY(timed("wgrad_gate_up", s, [&] { return launch_lora_wgrad_tc(wp, 2, L.rp, r, rt->offsets, E, N, dev_status, s); }));
    }
    return MOE_OK;
}

moe_status moe_lora_fwd(const moe_dims* d, const moe_routing* rt, const uint16_t* x, const uint16_t* W_gu,
                        const uint16_t* A_gu, const uint16_t* B_gu, const uint16_t* W_d, const uint16_t* A_d,
                        const uint16_t* B_d, uint16_t* y, void* saved, size_t saved_bytes, void* workspace,
                        size_t workspace_bytes, int32_t* dev_status, void* stream) {
    return fwd_impl(d, rt, x, W_gu, nullptr, A_gu, B_gu, W_d, nullptr, A_d, B_d, y, saved, saved_bytes, workspace,
                    workspace_bytes, dev_status, stream);
}

moe_status moe_lora_fwd_h_from_gu(const moe_dims* d, const moe_routing* rt, const uint16_t* x, const uint16_t* W_gu,
                                  const uint16_t* A_gu, const uint16_t* B_gu, const uint16_t* W_d, const uint16_t* A_d,
                                  const uint16_t* B_d, uint16_t* y, void* saved, size_t saved_bytes, void* workspace,
                                  size_t workspace_bytes, int32_t* dev_status, void* stream) {
    return fwd_impl(d, rt, x, W_gu, nullptr, A_gu, B_gu, W_d, nullptr, A_d, B_d, y, saved, saved_bytes, workspace,
                    workspace_bytes, dev_status, stream, 0, true);
}

moe_status moe_lora_bwd(const moe_dims* d, const moe_routing* rt, const uint16_t* dy, const uint16_t* W_gu,
                        const uint16_t* A_gu, const uint16_t* B_gu, const uint16_t* W_d, const uint16_t* A_d,
                        const uint16_t* B_d, const void* saved, size_t saved_bytes, uint16_t* dx,
                        uint16_t* dA_gu, uint16_t* dB_gu, uint16_t* dA_d, uint16_t* dB_d, float* d_topk_w,
                        void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
    return bwd_impl(d, rt, dy, W_gu, nullptr, A_gu, B_gu, W_d, nullptr, A_d, B_d, saved, saved_bytes, dx, dA_gu,
                    dB_gu, dA_d, dB_d, d_topk_w, workspace, workspace_bytes, dev_status, stream);
}

moe_status moe_lora_fwd_fp8(const moe_dims* d, const moe_routing* rt, const uint16_t* x, const uint8_t* Wq_gu,
                            const float* s_gu, const uint16_t* A_gu, const uint16_t* B_gu, const uint8_t* Wq_d,
                            const float* s_d, const uint16_t* A_d, const uint16_t* B_d, uint16_t* y, void* saved,
                            size_t saved_bytes, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                            void* stream) {
    if (s_gu == nullptr || s_d == nullptr) return MOE_ERR_NULL_ARG;
    return fwd_impl(d, rt, x, Wq_gu, s_gu, A_gu, B_gu, Wq_d, s_d, A_d, B_d, y, saved, saved_bytes, workspace,
                    workspace_bytes, dev_status, stream, 8);
}

moe_status moe_lora_bwd_fp8(const moe_dims* d, const moe_routing* rt, const uint16_t* dy, const uint8_t* Wq_gu,
                            const float* s_gu, const uint16_t* A_gu, const uint16_t* B_gu, const uint8_t* Wq_d,
                            const float* s_d, const uint16_t* A_d, const uint16_t* B_d, const void* saved,
                            size_t saved_bytes, uint16_t* dx, uint16_t* dA_gu, uint16_t* dB_gu, uint16_t* dA_d,
                            uint16_t* dB_d, float* d_topk_w, void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, void* stream) {
    if (s_gu == nullptr || s_d == nullptr) return MOE_ERR_NULL_ARG;
    return bwd_impl(d, rt, dy, Wq_gu, s_gu, A_gu, B_gu, Wq_d, s_d, A_d, B_d, saved, saved_bytes, dx, dA_gu, dB_gu,
                    dA_d, dB_d, d_topk_w, workspace, workspace_bytes, dev_status, stream, 8);
}

moe_status moe_lora_fwd_nf4(const moe_dims* d, const moe_routing* rt, const uint16_t* x, const uint8_t* Wq_gu,
                            const float* absmax_gu, const uint16_t* A_gu, const uint16_t* B_gu, const uint8_t* Wq_d,
                            const float* absmax_d, const uint16_t* A_d, const uint16_t* B_d, uint16_t* y, void* saved,
                            size_t saved_bytes, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                            void* stream) {
    if (absmax_gu == nullptr || absmax_d == nullptr) return MOE_ERR_NULL_ARG;
    return fwd_impl(d, rt, x, Wq_gu, absmax_gu, A_gu, B_gu, Wq_d, absmax_d, A_d, B_d, y, saved, saved_bytes,
                    workspace, workspace_bytes, dev_status, stream, 4);
}

moe_status moe_lora_bwd_nf4(const moe_dims* d, const moe_routing* rt, const uint16_t* dy, const uint8_t* Wq_gu,
                            const float* absmax_gu, const uint16_t* A_gu, const uint16_t* B_gu, const uint8_t* Wq_d,
                            const float* absmax_d, const uint16_t* A_d, const uint16_t* B_d, const void* saved,
                            size_t saved_bytes, uint16_t* dx, uint16_t* dA_gu, uint16_t* dB_gu, uint16_t* dA_d,
                            uint16_t* dB_d, float* d_topk_w, void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, void* stream) {
    if (absmax_gu == nullptr || absmax_d == nullptr) return MOE_ERR_NULL_ARG;
    return bwd_impl(d, rt, dy, Wq_gu, absmax_gu, A_gu, B_gu, Wq_d, absmax_d, A_d, B_d, saved, saved_bytes, dx, dA_gu,
                    dB_gu, dA_d, dB_d, d_topk_w, workspace, workspace_bytes, dev_status, stream, 4);
}

moe_status moe_quantize_fp8(const uint16_t* W, int64_t n_mat, int64_t rows, int32_t cols, uint8_t* Wq,
                            float* scales, void* stream) {
    if (n_mat < 0 || rows < 0 || cols < 0) return MOE_ERR_BAD_DIMS;
    if (n_mat * rows * (int64_t)cols > 0 && (W == nullptr || Wq == nullptr || scales == nullptr))
        return MOE_ERR_NULL_ARG;
    if (!aligned16(W) || !aligned16(Wq) || !aligned16(scales)) return MOE_ERR_MISALIGNED;
    return cuda_status(timed("quantize_fp8", (cudaStream_t)stream, [&] {
        return launch_quantize_fp8(W, n_mat, rows, cols, Wq, scales, (cudaStream_t)stream);
    }));
}

moe_status moe_quantize_nf4(const uint16_t* W, int64_t n_mat, int64_t rows, int32_t cols, uint8_t* Wq,
                            float* absmax, void* stream) {
    if (n_mat < 0 || rows < 0 || cols < 0 || cols % 64 != 0) return MOE_ERR_BAD_DIMS;
    if (n_mat * rows * (int64_t)cols > 0 && (W == nullptr || Wq == nullptr || absmax == nullptr))
        return MOE_ERR_NULL_ARG;
    if (!aligned16(W) || !aligned16(Wq) || !aligned16(absmax)) return MOE_ERR_MISALIGNED;
    return cuda_status(timed("quantize_nf4", (cudaStream_t)stream, [&] {
        return launch_quantize_nf4(W, n_mat, rows, cols, Wq, absmax, (cudaStream_t)stream);
    }));
}

moe_status moe_nf4_codebook(float* values) {
    if (values == nullptr) return MOE_ERR_NULL_ARG;
    memcpy(values, nf4_table().v, sizeof(nf4_table().v));
    return MOE_OK;
}

moe_status moe_router_topk(const float* logits, int64_t T, int32_t E, int32_t k, int32_t* topk_idx, float* topk_w,
                           void* stream) {
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E || T * (int64_t)k >= (int64_t(1) << 31)) return MOE_ERR_BAD_DIMS;
    if (T > 0 && (logits == nullptr || topk_idx == nullptr || topk_w == nullptr)) return MOE_ERR_NULL_ARG;
    if (!aligned16(logits) || !aligned16(topk_idx) || !aligned16(topk_w)) return MOE_ERR_MISALIGNED;
    return cuda_status(timed("router_topk", (cudaStream_t)stream, [&] {
        return launch_router_topk(logits, T, E, k, topk_idx, topk_w, (cudaStream_t)stream);
    }, T > 0 ? 1 : 0));
}

moe_status moe_router_bwd(const float* logits, const int32_t* topk_idx, const float* d_topk_w, int64_t T, int32_t E,
                          int32_t k, float* d_logits, void* stream) {
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E || T * (int64_t)k >= (int64_t(1) << 31)) return MOE_ERR_BAD_DIMS;
    if (T > 0 && (logits == nullptr || topk_idx == nullptr || d_topk_w == nullptr || d_logits == nullptr))
        return MOE_ERR_NULL_ARG;
    if (!aligned16(logits) || !aligned16(topk_idx) || !aligned16(d_topk_w) || !aligned16(d_logits))
        return MOE_ERR_MISALIGNED;
    return cuda_status(timed("router_bwd", (cudaStream_t)stream, [&] {
        return launch_router_bwd(logits, topk_idx, d_topk_w, T, E, k, d_logits, (cudaStream_t)stream);
    }, T > 0 ? 1 : 0));
}

// Packed batches of up to 2^30 tokens: the kernels' token indices (and a chunk past the
// last token) stay within int32.
constexpr int64_t kPackedMaxTokens = int64_t(1) << 30;

moe_status moe_packed_metadata(const void* position_ids, int32_t pos_bytes, int64_t T, int32_t* cu_seqlens,
                               int32_t* seq_id, int32_t* n_seqs, int32_t* max_seqlen, void* stream) {
    if (T < 0 || T > kPackedMaxTokens || (pos_bytes != 4 && pos_bytes != 8)) return MOE_ERR_BAD_DIMS;
    if (cu_seqlens == nullptr || n_seqs == nullptr || max_seqlen == nullptr) return MOE_ERR_NULL_ARG;
    if (T > 0 && (position_ids == nullptr || seq_id == nullptr)) return MOE_ERR_NULL_ARG;
    const uintptr_t pw = (uintptr_t)position_ids;
    if ((pw & (uintptr_t)(pos_bytes - 1)) != 0) return MOE_ERR_MISALIGNED;
    for (const void* p : {(const void*)cu_seqlens, (const void*)seq_id, (const void*)n_seqs, (const void*)max_seqlen})
        if (((uintptr_t)p & 3u) != 0) return MOE_ERR_MISALIGNED;
    return cuda_status(timed("packed_meta", (cudaStream_t)stream, [&] {
        return launch_packed_metadata(position_ids, pos_bytes, T, cu_seqlens, seq_id, n_seqs, max_seqlen,
                                      (cudaStream_t)stream);
    }));
}

moe_status moe_packed_causal_mask(const int32_t* cu_seqlens, const int32_t* seq_id, int64_t T, uint8_t* mask,
                                  void* stream) {
    if (T < 0 || T > kPackedMaxTokens) return MOE_ERR_BAD_DIMS;
    if (T > 0 && (cu_seqlens == nullptr || seq_id == nullptr || mask == nullptr)) return MOE_ERR_NULL_ARG;
    if (((uintptr_t)cu_seqlens & 3u) != 0 || ((uintptr_t)seq_id & 3u) != 0 || !aligned16(mask))
        return MOE_ERR_MISALIGNED;
    return cuda_status(timed("packed_mask", (cudaStream_t)stream, [&] {
        return launch_packed_mask(cu_seqlens, seq_id, T, mask, (cudaStream_t)stream);
    }, T > 0 ? 1 : 0));
}

moe_status moe_diag_force_timeout(int32_t launch_index, uint64_t limit_ns) {
    ForcedTimeout& f = forced();
    if (launch_index < 0) {
        f.target.store(-1);
        return MOE_OK;
    }
    if (limit_ns < 1000 || limit_ns > tc::kWaitTimeoutNs) return MOE_ERR_BAD_DIMS;
    f.target.store(-1);
    f.limit_ns.store(limit_ns);
    f.seen.store(0);
    f.target.store(launch_index);
    return MOE_OK;
}

moe_status moe_timing_enable(int32_t on) {
    Timing& t = timing();
    std::lock_guard<std::mutex> g(t.mu);
    t.on = on != 0;
    if (t.on) t.used = 0;      // enabling starts a new record; disabling keeps it for moe_timing_read
    return MOE_OK;
}

moe_status moe_timing_read(int32_t index, char* name, size_t name_len, double* total_ms, int32_t* launches) {
    if (name == nullptr || total_ms == nullptr || launches == nullptr || name_len == 0) return MOE_ERR_NULL_ARG;
    Timing& t = timing();
    std::lock_guard<std::mutex> g(t.mu);
    // distinct names in first-seen order
    std::vector<const char*> names;
    for (size_t i = 0; i < t.used; ++i) {
        bool seen = false;
        for (const char* n : names) seen = seen || strcmp(n, t.pool[i].name) == 0;
        if (!seen) names.push_back(t.pool[i].name);
    }
    if (index < 0 || (size_t)index >= names.size()) return MOE_ERR_BAD_DIMS;
    double ms = 0.0;
    int32_t n = 0;
    for (size_t i = 0; i < t.used; ++i) {
        if (strcmp(t.pool[i].name, names[index]) != 0) continue;
        if (cudaEventSynchronize(t.pool[i].stop) != cudaSuccess) return MOE_ERR_CUDA;
        float e = 0.f;
        if (cudaEventElapsedTime(&e, t.pool[i].start, t.pool[i].stop) != cudaSuccess) return MOE_ERR_CUDA;
        ms += e;
        ++n;
    }
    strncpy(name, names[index], name_len - 1);
    name[name_len - 1] = 0;
    *total_ms = ms;
    *launches = n;
    return MOE_OK;
}

uint64_t moe_launch_count(void) {
    Timing& t = timing();
    std::lock_guard<std::mutex> g(t.mu);
    return t.launches;
}

}  // extern "C"
