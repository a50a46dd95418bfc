// C ABI of libmoefp8.so (declared in include/moe_fp8.h): argument checks,
// workspace layout and the forward pass as one stream-ordered sequence.
#include <atomic>
#include <cstring>

#include "common.cuh"

namespace moe {

namespace {
thread_local int g_last_cuda_error = 0;
std::atomic<uint64_t> g_launches{0};
constexpr long long kDefaultWaitCycles = 4000000000LL;   // about 2 s of SM clock
std::atomic<long long> g_wait_cycles{kDefaultWaitCycles};
std::atomic<int> g_stall{0};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Workspace layout shared by moe_forward, moe_route and moe_permute.
struct Layout {
    size_t status, route, hist, base, go, offsets, perm, inv_row, A, sa, H, sh, Y, Ysh, total;
};

Layout layout(int T, int d, int E, int K, int S, int I) {
    Layout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    const size_t M = (size_t)T * (K + S);
    const size_t nchunks = ((size_t)T + kPermuteChunk - 1) / kPermuteChunk;
    L.status = take(16);
    L.route = take(route_ws_bytes(T, d, E));
    L.hist = take(sizeof(int32_t) * nchunks * E);
    L.base = take(sizeof(int32_t) * nchunks * E);
    L.go = take(sizeof(int32_t) * (size_t)(E + S + 1));
    L.offsets = take(sizeof(int32_t) * (size_t)(E + 1));
    L.perm = take(sizeof(int32_t) * M);
    L.inv_row = take(sizeof(int32_t) * (size_t)T * K);
    L.A = take(M * d);
    L.sa = take(sizeof(float) * M * (d / 128));
    L.H = take(M * I);
    L.sh = take(sizeof(float) * M * (I / 128));
    // routed expert outputs in bf16; the shared experts' (weight 1 in h') in float32
    L.Y = take(sizeof(uint16_t) * (size_t)T * K * d);
    L.Ysh = take(sizeof(float) * (size_t)T * S * d);
    L.total = off;
    return L;
}

// Group-limited routing parameters (n_groups = 0 means plain top-K when allowed).
int check_groups(int E, int K, int n_groups, int topk_groups, int group_topk, bool zero_ok) {
    if (n_groups == 0 && zero_ok) return MOE_OK;
    if (n_groups < 1 || n_groups > 32 || E % n_groups) return MOE_ERR_INVALID_ARG;
    const int gs = E / n_groups;
    if (topk_groups < 1 || topk_groups > n_groups || group_topk < 1 || group_topk > gs)
        return MOE_ERR_INVALID_ARG;
    if (K > topk_groups * gs) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

int check_layer(const moe_layer_t* L) {
    if (!L) return MOE_ERR_INVALID_ARG;
    if (L->d <= 0 || L->E <= 0 || L->K <= 0 || L->S < 0 || L->I <= 0) return MOE_ERR_INVALID_ARG;
    if (L->E > kMaxExperts || L->K > kMaxTopK || L->K > L->E) return MOE_ERR_INVALID_ARG;
    // the dispatch quantiser gives each of a token's K + S rows its own lane
    if (L->K + L->S > 32) return MOE_ERR_INVALID_ARG;
    if (L->d % 128 || L->I % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (L->E + L->S > kMaxGroups) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!L->centroids || !L->bias || !L->w_gate || !L->w_up || !L->w_down || !L->s_gate ||
        !L->s_up || !L->s_down)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(L->centroids) || !aligned16(L->w_gate) || !aligned16(L->w_up) ||
        !aligned16(L->w_down))
        return MOE_ERR_MISALIGNED;
    return check_groups(L->E, L->K, L->n_groups, L->topk_groups, L->group_topk, true);
}

inline cudaStream_t S_(void* s) { return static_cast<cudaStream_t>(s); }

// Batches of at most this many tokens run the gate/up GEMM, and of at most
// kSmallDownT tokens the down GEMM, with the small-group tiles (measured on
// B300 with the V3 decode shapes: gate/up 60 vs 74 us at T = 1, 888 vs 903 us
// at T = 64; down equal at T = 1 to 4, slower with the small tiles from T = 16).
constexpr int kSmallGemmT = 64;
constexpr int kSmallDownT = 4;

int launch_gemm_large(int mode, const uint8_t* A, const float* sa, int M_total, const int32_t* go,
                      int G, const uint8_t* W0, const uint8_t* W1, const float* sw0,
                      const float* sw1, int N, int Kdim, void* out, float* out_scales,
                      int32_t* status, cudaStream_t st, int f32_group0, int f32_row0, float* out2,
                      int counter_slot, bool counter_zeroed, int max_ctas) {
    return launch_grouped_gemm(mode, A, sa, M_total, go, G, W0, W1, sw0, sw1, N, Kdim, out,
                               out_scales, status, st, nullptr, f32_group0, f32_row0, out2,
                               counter_slot, counter_zeroed, max_ctas);
}

}  // namespace

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

long long pipeline_wait_cycles() { return g_wait_cycles.load(std::memory_order_relaxed); }
int pipeline_stall() { return g_stall.load(std::memory_order_relaxed); }

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return MOE_ERR_CUDA;
}

int check_launch() {
    note_launch();
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case MOE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_TIMEOUT: return "GEMM pipeline wait timed out";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_BAD_INDEX: return "index out of range in device data";
        default: return "unknown status";
    }
}

int moe_last_cuda_error(void) { return g_last_cuda_error; }

uint64_t moe_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

long long moe_set_pipeline_wait_limit(long long cycles) {
    return g_wait_cycles.exchange(cycles > 0 ? cycles : kDefaultWaitCycles);
}

int moe_set_pipeline_stall(int on) { return g_stall.exchange(on ? 1 : 0); }

size_t moe_workspace_size(const moe_layer_t* L, int T_max) {
    if (!L || T_max < 0 || L->d <= 0 || L->E <= 0 || L->K <= 0 || L->S < 0 || L->I <= 0) return 0;
    return layout(T_max, L->d, L->E, L->K, L->S, L->I).total;
}

int moe_quant_1x128(const uint16_t* x, int n_src, const int32_t* gather_rows, int M, int d,
                    uint8_t* q, float* scales, int scale_ld, int32_t* status, void* stream) {
    if (M < 0 || n_src < 0 || d <= 0 || scale_ld < M) return MOE_ERR_INVALID_ARG;
    if (d % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return MOE_OK;
    if (!x || !q || !scales) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q)) return MOE_ERR_MISALIGNED;
    // every output row is a gathered row (no shared-expert tail)
    return launch_quant_1x128(x, n_src, gather_rows, /*n_gather=*/M, /*tail_T=*/1, M, d, q, scales,
                              scale_ld, status, S_(stream));
}

int moe_quant_1x128_dispatch(const uint16_t* x, int T, int d, const int32_t* inv_row, int K,
                             int S, uint8_t* q, float* scales, int scale_ld, int32_t* status,
                             void* stream) {
    if (T < 0 || d <= 0 || K < 0 || S < 0 || K + S > 32 || K + S == 0) return MOE_ERR_INVALID_ARG;
    if (d % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((long long)T * (K + S) > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (scale_ld < T * (K + S)) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !q || !scales || (K > 0 && !inv_row)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q)) return MOE_ERR_MISALIGNED;
    return launch_quant_dispatch(x, T, d, inv_row, K, S, q, scales, scale_ld, status, S_(stream));
}

int moe_quant_128x128(const float* w, int R, int C, uint8_t* q, float* scales, void* stream) {
    if (R < 0 || C < 0) return MOE_ERR_INVALID_ARG;
    if (R % 128 || C % 128 || R / 128 > 65535) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (R == 0 || C == 0) return MOE_OK;
    if (!w || !q || !scales) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(q)) return MOE_ERR_MISALIGNED;
    return launch_quant_128x128(w, R, C, q, scales, S_(stream));
}

size_t moe_route_workspace_size(int T, int d, int E) {
    if (T < 0 || d <= 0 || E <= 0 || d % 128 || E > kMaxExperts) return 0;
    return route_ws_bytes(T, d, E);
}

int moe_route_estimate_logits(const uint16_t* u, const float* centroids, int T, int d, int E,
                              float* logits, float* norms, void* ws, size_t ws_bytes,
                              void* stream) {
    if (T < 0 || d <= 0 || E <= 0 || E > kMaxExperts) return MOE_ERR_INVALID_ARG;
    if (d % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    if (!u || !centroids || !logits || !norms || !ws) return MOE_ERR_INVALID_ARG;
    if (!aligned16(u) || !aligned16(centroids)) return MOE_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_MISALIGNED;
    if (ws_bytes < route_ws_bytes(T, d, E)) return MOE_ERR_WORKSPACE;
    int32_t* status = static_cast<int32_t*>(ws);
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), S_(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return launch_route_estimate(u, centroids, T, d, E, logits, norms, ws, status, S_(stream));
}

int moe_route_grouped(const uint16_t* u, const float* centroids, const float* bias, int T, int d,
                      int E, int K, int n_groups, int topk_groups, int group_topk,
                      int32_t* topk_idx, float* topk_gate, uint8_t* tie_flag, int32_t* counts,
                      void* ws, size_t ws_bytes, void* stream) {
    if (T < 0 || d <= 0 || E <= 0 || K <= 0 || K > E || K > kMaxTopK || E > kMaxExperts)
        return MOE_ERR_INVALID_ARG;
    if (d % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    int rc = check_groups(E, K, n_groups, topk_groups, group_topk, false);
    if (rc) return rc;
    if (!counts || !centroids || !bias) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!u || !topk_idx || !topk_gate || !tie_flag || !ws)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(u) || !aligned16(centroids)) return MOE_ERR_MISALIGNED;
    if (T == 0) return launch_route_tc(u, centroids, bias, 0, d, E, K, topk_idx, topk_gate,
                                       tie_flag, counts, ws, nullptr, S_(stream));
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_MISALIGNED;
    if (ws_bytes < route_ws_bytes(T, d, E)) return MOE_ERR_WORKSPACE;
    int32_t* status = static_cast<int32_t*>(ws);
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), S_(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return launch_route_tc(u, centroids, bias, T, d, E, K, topk_idx, topk_gate, tie_flag, counts,
                           ws, status, S_(stream), n_groups, topk_groups, group_topk);
}

int moe_route(const uint16_t* u, const float* centroids, const float* bias, int T, int d, int E,
              int K, int32_t* topk_idx, float* topk_gate, uint8_t* tie_flag, int32_t* counts,
              void* ws, size_t ws_bytes, void* stream) {
    if (T < 0 || d <= 0 || E <= 0 || K <= 0 || K > E || K > kMaxTopK || E > kMaxExperts)
        return MOE_ERR_INVALID_ARG;
    if (d % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!counts || !centroids || !bias) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!u || !topk_idx || !topk_gate || !tie_flag || !ws)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(u) || !aligned16(centroids)) return MOE_ERR_MISALIGNED;
    if (T == 0) return launch_route_tc(u, centroids, bias, 0, d, E, K, topk_idx, topk_gate,
                                       tie_flag, counts, ws, nullptr, S_(stream));
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_MISALIGNED;
    if (ws_bytes < route_ws_bytes(T, d, E)) return MOE_ERR_WORKSPACE;
    // the workspace's first int32 is the status word of this call
    int32_t* status = static_cast<int32_t*>(ws);
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), S_(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return launch_route_tc(u, centroids, bias, T, d, E, K, topk_idx, topk_gate, tie_flag, counts,
                           ws, status, S_(stream));
}

int moe_permute(const int32_t* topk_idx, int T, int K, int E, int S, int32_t* offsets,
                int32_t* group_offsets, int32_t* perm_token, int32_t* inv_row, int32_t* status,
                void* ws, size_t ws_bytes, void* stream) {
    if (T < 0 || K <= 0 || E <= 0 || S < 0 || K > E || K > kMaxTopK || E > kMaxExperts)
        return MOE_ERR_INVALID_ARG;
    if ((long long)T * (K + S) > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!offsets || !ws || (T > 0 && (!topk_idx || !perm_token || !inv_row)))
        return MOE_ERR_INVALID_ARG;
    const size_t nchunks = ((size_t)T + kPermuteChunk - 1) / kPermuteChunk;
    const size_t hist_bytes = align_up(sizeof(int32_t) * nchunks * E, 256);
    if (ws_bytes < 2 * hist_bytes) return MOE_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_MISALIGNED;
    int32_t* hist = static_cast<int32_t*>(ws);
    int32_t* base = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + hist_bytes);
    return launch_permute(topk_idx, T, K, E, offsets, perm_token, inv_row, group_offsets, S,
                          status, hist, base, S_(stream));
}

int moe_grouped_gemm_fp8(int mode, const uint8_t* A, const float* sa, int M_total,
                         const int32_t* group_offsets, int G, const uint8_t* W0,
                         const uint8_t* W1, const float* sw0, const float* sw1, int N, int Kdim,
                         void* out, float* out_scales, int32_t* status, void* stream) {
    if (mode != MOE_GEMM_GATE_UP_SILU_QUANT && mode != MOE_GEMM_DOWN && mode != MOE_GEMM_DOWN_F32)
        return MOE_ERR_INVALID_ARG;
    if (M_total < 0 || G < 0 || N <= 0 || Kdim <= 0) return MOE_ERR_INVALID_ARG;
    if (N % 128 || Kdim % 128 || G > kMaxGroups) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((long long)G * N > 0x7fffffffLL || (long long)M_total * (N > Kdim ? N : Kdim) > (1LL << 40))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (M_total == 0 || G == 0) return MOE_OK;
    if (!A || !sa || !group_offsets || !W0 || !sw0 || !out) return MOE_ERR_INVALID_ARG;
    const bool gu = mode == MOE_GEMM_GATE_UP_SILU_QUANT;
    if (gu && (!W1 || !sw1 || !out_scales)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(W0) || (gu && !aligned16(W1)) || !aligned16(out))
        return MOE_ERR_MISALIGNED;
    return launch_grouped_gemm(mode, A, sa, M_total, group_offsets, G, W0, W1, sw0, sw1, N, Kdim,
                               out, out_scales, status, S_(stream));
}

int moe_grouped_gemm_fp8_small(int mode, const uint8_t* A, const float* sa, int M_total,
                               const int32_t* group_offsets, int G, const uint8_t* W0,
                               const uint8_t* W1, const float* sw0, const float* sw1, int N,
                               int Kdim, void* out, float* out_scales, int32_t* status,
                               void* stream) {
    if (mode != MOE_GEMM_GATE_UP_SILU_QUANT && mode != MOE_GEMM_DOWN && mode != MOE_GEMM_DOWN_F32)
        return MOE_ERR_INVALID_ARG;
    if (M_total < 0 || G < 0 || N <= 0 || Kdim <= 0) return MOE_ERR_INVALID_ARG;
    if (N % 128 || Kdim % 128 || G > kMaxGroups) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((long long)G * N > 0x7fffffffLL || (long long)M_total * (N > Kdim ? N : Kdim) > (1LL << 40))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (M_total == 0 || G == 0) return MOE_OK;
    if (!A || !sa || !group_offsets || !W0 || !sw0 || !out) return MOE_ERR_INVALID_ARG;
    const bool gu = mode == MOE_GEMM_GATE_UP_SILU_QUANT;
    if (gu && (!W1 || !sw1 || !out_scales)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(W0) || (gu && !aligned16(W1)) || !aligned16(out))
        return MOE_ERR_MISALIGNED;
    return launch_grouped_gemm_small(mode, A, sa, M_total, group_offsets, G, W0, W1, sw0, sw1, N,
                                     Kdim, out, out_scales, status, S_(stream));
}

int moe_grouped_gemm_fp8_down(const uint8_t* H, const float* sh, int M_total,
                              const int32_t* group_offsets, int G, int f32_group0, int f32_row0,
                              const uint8_t* W, const float* sw, int N, int Kdim, uint16_t* y,
                              float* y_f32, int small_tiles, int32_t* status, void* stream) {
    if (M_total < 0 || G < 0 || N <= 0 || Kdim <= 0 || f32_group0 < 0 || f32_row0 < 0)
        return MOE_ERR_INVALID_ARG;
    if (N % 128 || Kdim % 128 || G > kMaxGroups) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((long long)G * N > 0x7fffffffLL || (long long)M_total * (N > Kdim ? N : Kdim) > (1LL << 40))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (M_total == 0 || G == 0) return MOE_OK;
    if (!H || !sh || !group_offsets || !W || !sw) return MOE_ERR_INVALID_ARG;
    if ((f32_group0 > 0 && !y) || (f32_group0 < G && !y_f32)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(H) || !aligned16(W) || !aligned16(y) || !aligned16(y_f32)) return MOE_ERR_MISALIGNED;
    const auto gemm = small_tiles ? launch_grouped_gemm_small : launch_gemm_large;
    return gemm(MOE_GEMM_DOWN, H, sh, M_total, group_offsets, G, W, nullptr, sw, nullptr, N, Kdim,
                y, nullptr, status, S_(stream), f32_group0, f32_row0, y_f32, 1, false, 0);
}

int moe_combine(const uint16_t* u, const uint16_t* Y, const float* topk_gate,
                const int32_t* inv_row, const float* Y_shared, int T, int d, int K, int S,
                float* h_out, void* stream) {
    if (T < 0 || d <= 0 || K < 0 || K > kMaxTopK || S < 0) return MOE_ERR_INVALID_ARG;
    if (d % 8) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    if (!u || !h_out || (K > 0 && (!Y || !topk_gate || !inv_row)) || (S > 0 && !Y_shared))
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(u) || !aligned16(Y) || !aligned16(Y_shared) || !aligned16(h_out))
        return MOE_ERR_MISALIGNED;
    return launch_combine(u, Y, topk_gate, inv_row, Y_shared, T, d, K, S, h_out, S_(stream));
}

}  // extern "C"

namespace moe {
namespace {

// Pointers of one forward's workspace (the layout above).
struct Fwd {
    int32_t *status, *hist, *bbase, *go, *offsets, *perm, *inv_row;
    void* route_ws;
    uint8_t *A, *H;
    float *sa, *sh, *Ysh;
    uint16_t* Y;
};

Fwd fwd_ptrs(const moe_layer_t* L, int T, void* ws) {
    const Layout W = layout(T, L->d, L->E, L->K, L->S, L->I);
    char* base = static_cast<char*>(ws);
    Fwd f;
    f.status = reinterpret_cast<int32_t*>(base + W.status);
    f.route_ws = base + W.route;
    f.hist = reinterpret_cast<int32_t*>(base + W.hist);
    f.bbase = reinterpret_cast<int32_t*>(base + W.base);
    f.go = reinterpret_cast<int32_t*>(base + W.go);
    f.offsets = reinterpret_cast<int32_t*>(base + W.offsets);
    f.perm = reinterpret_cast<int32_t*>(base + W.perm);   // T*(K+S) rows
    f.inv_row = reinterpret_cast<int32_t*>(base + W.inv_row);
    f.A = reinterpret_cast<uint8_t*>(base + W.A);
    f.sa = reinterpret_cast<float*>(base + W.sa);
    f.H = reinterpret_cast<uint8_t*>(base + W.H);
    f.sh = reinterpret_cast<float*>(base + W.sh);
    f.Y = reinterpret_cast<uint16_t*>(base + W.Y);
    f.Ysh = reinterpret_cast<float*>(base + W.Ysh);
    return f;
}

// Host-side checks shared by the forward entry points.
int check_forward(const moe_layer_t* L, const uint16_t* u, int T, float* h_out, int32_t* topk_idx,
                  float* topk_gate, int32_t* counts, uint8_t* tie_flag, void* ws, size_t ws_bytes) {
    int rc = check_layer(L);
    if (rc) return rc;
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if ((long long)T * (L->K + L->S) > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!ws || !counts) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!u || !h_out || !topk_idx || !topk_gate || !tie_flag)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(u) || !aligned16(h_out)) return MOE_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_MISALIGNED;
    if (ws_bytes < layout(T, L->d, L->E, L->K, L->S, L->I).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

// Phase 1 of a forward: status word, routing, dispatch, quantisation.
// reset_status = false keeps status[0] (the device errors of earlier calls);
// status[1] and status[2], the two GEMMs' tile counters, are always zeroed
// here, so that no memset sits between the layer's kernels.
int forward_prep(const moe_layer_t* L, const uint16_t* u, int T, int32_t* topk_idx,
                 float* topk_gate, int32_t* counts, uint8_t* tie_flag, const Fwd& f,
                 cudaStream_t st, bool reset_status) {
    const int d = L->d, E = L->E, K = L->K, S = L->S;
    int rc;
    const cudaError_t e = reset_status ? cudaMemsetAsync(f.status, 0, 16, st)
                                       : cudaMemsetAsync(f.status + 1, 0, 12, st);
    if (e != cudaSuccess) return cuda_fail(e);
    if ((rc = launch_route_layer(u, L->centroids, L->bias, T, d, E, K, topk_idx, topk_gate, tie_flag,
                                 counts, f.route_ws, f.status, st, L->n_groups, L->topk_groups,
                                 L->group_topk)))
        return rc;
    if (T == 0) return MOE_OK;
    if ((rc = launch_permute(topk_idx, T, K, E, f.offsets, f.perm, f.inv_row, f.go, S, f.status,
                             f.hist, f.bbase, st)))
        return rc;
    return launch_quant_dispatch(u, T, d, f.inv_row, K, S, f.A, f.sa, T * (K + S), f.status, st);
}

// Phase 2: the two expert GEMMs (max_ctas > 0 caps their persistent grids).
int forward_gemms(const moe_layer_t* L, int T, const Fwd& f, cudaStream_t st, int max_ctas) {
    if (T == 0) return MOE_OK;
    const int d = L->d, E = L->E, K = L->K, S = L->S, I = L->I, G = E + S;
    const int M = T * (K + S);
    // Few tokens: no group has more than T rows, so the weight panels dominate
    // the bytes and the tiles of 128 weight rows x 32 rows keep more of them in
    // flight per SM (gemm_small.cu).  Routed rows of y in bf16, shared rows
    // (weight 1 in h') in float32.
    const auto gemm = T <= kSmallGemmT ? launch_grouped_gemm_small : launch_gemm_large;
    const auto gemm_down = T <= kSmallDownT ? launch_grouped_gemm_small : launch_gemm_large;
    int rc;
    if ((rc = gemm(MOE_GEMM_GATE_UP_SILU_QUANT, f.A, f.sa, M, f.go, G, L->w_gate, L->w_up,
                   L->s_gate, L->s_up, I, d, f.H, f.sh, f.status, st, 1 << 30, 0, nullptr, 1, true,
                   max_ctas)))
        return rc;
    // routed groups' rows (the first T*K) to Y in bf16, shared groups' rows to Ysh in float32
    return gemm_down(MOE_GEMM_DOWN, f.H, f.sh, M, f.go, G, L->w_down, nullptr, L->s_down, nullptr, d,
                     I, f.Y, nullptr, f.status, st, E, T * K, f.Ysh, 2, true, max_ctas);
}

// Phase 3: h' = u + shared + gated routed outputs.
int forward_combine(const moe_layer_t* L, const uint16_t* u, int T, const float* topk_gate,
                    float* h_out, const Fwd& f, cudaStream_t st) {
    if (T == 0) return MOE_OK;
    return launch_combine(u, f.Y, topk_gate, f.inv_row, f.Ysh, T, L->d, L->K, L->S, h_out, st);
}

// moe_forward's body; reset_status = false keeps the status word of earlier
// calls (moe_forward_host clears it once for its whole batch sequence).
int forward_impl(const moe_layer_t* L, const uint16_t* u, int T, float* h_out, int32_t* topk_idx,
                 float* topk_gate, int32_t* counts, uint8_t* tie_flag, void* ws, size_t ws_bytes,
                 cudaStream_t st, bool reset_status) {
    int rc = check_forward(L, u, T, h_out, topk_idx, topk_gate, counts, tie_flag, ws, ws_bytes);
    if (rc) return rc;
    const Fwd f = fwd_ptrs(L, T, ws);
    if ((rc = forward_prep(L, u, T, topk_idx, topk_gate, counts, tie_flag, f, st, reset_status)))
        return rc;
    if ((rc = forward_gemms(L, T, f, st, 0))) return rc;
    return forward_combine(L, u, T, topk_gate, h_out, f, st);
}

// Backward workspace: status, dy codes and scales, dH, [dG | dU] codes and
// scales, dA.
struct BwdLayout {
    size_t status, dyq, sdy, dH, dgu, sgu, dA, total;
};

BwdLayout bwd_layout(int T, int d, int K, int S, int I) {
    BwdLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    const size_t M = (size_t)T * (K + S);
    L.status = take(16);
    L.dyq = take(M * d);
    L.sdy = take(sizeof(float) * M * (d / 128));
    L.dH = take(sizeof(uint16_t) * M * I);
    L.dgu = take(M * 2 * I);
    L.sgu = take(sizeof(float) * M * (2 * I / 128));
    L.dA = take(sizeof(uint16_t) * M * d);
    L.total = off;
    return L;
}

// The re-quantised operands of the weight gradient (128x1 tiles, padded
// layout of moe_requant_128x1): ld columns each, scales [ld/128, C].
struct WgLayout {
    long long ld;
    size_t at, sat, ht, sht, dyt, sdyt, gut, sgut, total;
};

WgLayout wg_layout(int T, int d, int G, int K, int S, int I) {
    WgLayout L{};
    const long long M = (long long)T * (K + S);
    L.ld = (M + 127LL * G + 127) / 128 * 128;
    if (L.ld > 0x7fffffffLL) {
        L.ld = -1;
        return L;
    }
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    const size_t ld = (size_t)L.ld, nsl = ld / 128;
    L.at = take(ld * d);
    L.sat = take(sizeof(float) * nsl * d);
    L.ht = take(ld * I);
    L.sht = take(sizeof(float) * nsl * I);
    L.dyt = take(ld * d);
    L.sdyt = take(sizeof(float) * nsl * d);
    L.gut = take(ld * 2 * I);
    L.sgut = take(sizeof(float) * nsl * 2 * I);
    L.total = off;
    return L;
}

struct EventSet {
    cudaEvent_t ev[6] = {};
    ~EventSet() {
        for (cudaEvent_t e : ev)
            if (e) cudaEventDestroy(e);   // released when their last record completes
    }
};

}  // namespace
}  // namespace moe

extern "C" {

int moe_forward(const moe_layer_t* L, const uint16_t* u, int T, float* h_out, int32_t* topk_idx,
                float* topk_gate, int32_t* counts, uint8_t* tie_flag, void* ws, size_t ws_bytes,
                void* stream) {
    return forward_impl(L, u, T, h_out, topk_idx, topk_gate, counts, tie_flag, ws, ws_bytes,
                        S_(stream), true);
}

size_t moe_backward_workspace_size(const moe_layer_t* L, int T_max) {
    if (check_layer(L) || T_max < 0) return 0;
    return bwd_layout(T_max, L->d, L->K, L->S, L->I).total;
}

int moe_prepare_backward_weights(const moe_layer_t* L, uint8_t* w_down_t, float* s_down_t,
                                 uint8_t* w_gu_t, float* s_gu_t, void* stream) {
    int rc = check_layer(L);
    if (rc) return rc;
    if (!w_down_t || !s_down_t || !w_gu_t || !s_gu_t) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w_down_t) || !aligned16(w_gu_t)) return MOE_ERR_MISALIGNED;
    const int G = L->E + L->S, d = L->d, I = L->I;
    const cudaStream_t st = S_(stream);
    // W_down [G, d, I] -> W_down^T [G, I, d]
    if ((rc = launch_transpose_blocks(L->w_down, L->s_down, G, d, I, w_down_t, d, 0, s_down_t,
                                      d / 128, 0, st)))
        return rc;
    // W_gate, W_up [G, I, d] -> [W_gate^T | W_up^T] [G, d, 2I]
    if ((rc = launch_transpose_blocks(L->w_gate, L->s_gate, G, I, d, w_gu_t, 2 * I, 0, s_gu_t,
                                      2 * I / 128, 0, st)))
        return rc;
    return launch_transpose_blocks(L->w_up, L->s_up, G, I, d, w_gu_t, 2 * I, I, s_gu_t, 2 * I / 128,
                                   I / 128, st);
}

int moe_backward_dgrad(const moe_layer_t* L, const moe_layer_bwd_t* B, const uint16_t* u,
                       const uint16_t* dh, int T, const int32_t* topk_idx, const float* topk_gate,
                       float* du, void* fwd_ws, size_t fwd_ws_bytes, void* bwd_ws,
                       size_t bwd_ws_bytes, void* stream) {
    int rc = check_layer(L);
    if (rc) return rc;
    if (!B || !B->w_down_t || !B->s_down_t || !B->w_gu_t || !B->s_gu_t) return MOE_ERR_INVALID_ARG;
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!u || !dh || !topk_idx || !topk_gate || !du || !fwd_ws || !bwd_ws) return MOE_ERR_INVALID_ARG;
    if (!aligned16(u) || !aligned16(dh) || !aligned16(du) || !aligned16(B->w_down_t) ||
        !aligned16(B->w_gu_t))
        return MOE_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(fwd_ws) | reinterpret_cast<uintptr_t>(bwd_ws)) & 255u)
        return MOE_ERR_MISALIGNED;
    if ((long long)T * (L->K + L->S) > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int d = L->d, E = L->E, K = L->K, S = L->S, I = L->I, G = E + S;
    const Layout W = layout(T, d, E, K, S, I);
    const BwdLayout BW = bwd_layout(T, d, K, S, I);
    if (fwd_ws_bytes < W.total || bwd_ws_bytes < BW.total) return MOE_ERR_WORKSPACE;
    char* fb = static_cast<char*>(fwd_ws);
    char* bb = static_cast<char*>(bwd_ws);
    const cudaStream_t st = S_(stream);
    int32_t* status = reinterpret_cast<int32_t*>(bb + BW.status);
    const int32_t* go = reinterpret_cast<const int32_t*>(fb + W.go);
    const int32_t* inv_row = reinterpret_cast<const int32_t*>(fb + W.inv_row);
    const uint8_t* A = reinterpret_cast<const uint8_t*>(fb + W.A);
    const float* sa = reinterpret_cast<const float*>(fb + W.sa);
    const uint16_t* Y = reinterpret_cast<const uint16_t*>(fb + W.Y);
    uint8_t* dyq = reinterpret_cast<uint8_t*>(bb + BW.dyq);
    float* sdy = reinterpret_cast<float*>(bb + BW.sdy);
    uint16_t* dH = reinterpret_cast<uint16_t*>(bb + BW.dH);
    uint8_t* dgu = reinterpret_cast<uint8_t*>(bb + BW.dgu);
    float* sgu = reinterpret_cast<float*>(bb + BW.sgu);
    uint16_t* dA = reinterpret_cast<uint16_t*>(bb + BW.dA);
    const int M = T * (K + S);
    cudaError_t e = cudaMemsetAsync(status, 0, 16, st);
    if (e != cudaSuccess) return cuda_fail(e);
    if ((rc = launch_quant_dy(dh, T, d, topk_gate, inv_row, K, S, dyq, sdy, M, status, st))) return rc;
    // dH = dy W_down
    if ((rc = launch_grouped_gemm(MOE_GEMM_DOWN, dyq, sdy, M, go, G, B->w_down_t, nullptr,
                                  B->s_down_t, nullptr, I, d, dH, nullptr, status, st)))
        return rc;
    // G, U recomputed; [dG | dU]
    if ((rc = launch_grouped_gemm(MOE_GEMM_GATE_UP_DGRAD, A, sa, M, go, G, L->w_gate, L->w_up,
                                  L->s_gate, L->s_up, I, d, dgu, sgu, status, st, dH)))
        return rc;
    // dA = [dG | dU] [W_gate ; W_up]
    if ((rc = launch_grouped_gemm(MOE_GEMM_DOWN, dgu, sgu, M, go, G, B->w_gu_t, nullptr, B->s_gu_t,
                                  nullptr, d, 2 * I, dA, nullptr, status, st)))
        return rc;
    // du = dh + sum of the token's rows of dA, then the gate term
    if ((rc = launch_combine(dh, dA, nullptr, inv_row, dA + (size_t)T * K * d, T, d, K, S, du, st)))
        return rc;
    return launch_gate_term(u, dh, Y, inv_row, topk_idx, topk_gate, L->centroids, T, d, K, M, du,
                            status, st);
}

int moe_wgrad_ld(int M, int G) {
    if (M < 0 || G < 0) return 0;
    const long long ld = ((long long)M + 127LL * G + 127) / 128 * 128;
    return ld > 0x7fffffffLL ? 0 : (int)ld;
}

int moe_requant_128x1(const uint8_t* q, const float* scales, int M, int C,
                      const int32_t* group_offsets, int G, uint8_t* qt, float* st, int ld,
                      int32_t* status, void* stream) {
    if (M < 0 || C <= 0 || G < 0 || ld < 0) return MOE_ERR_INVALID_ARG;
    if (C % 128 || G > kMaxGroups || ld % 16) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (M == 0 || G == 0) return MOE_OK;
    if (!q || !scales || !group_offsets || !qt || !st) return MOE_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(qt)) return MOE_ERR_MISALIGNED;
    if ((long long)M * C > (1LL << 40) || (long long)ld * C > (1LL << 40)) return MOE_ERR_UNSUPPORTED_SHAPE;
    return launch_requant_128x1(q, scales, M, C, group_offsets, G, qt, st, ld, status, S_(stream));
}

int moe_wgrad_gemm_fp8(const uint8_t* At, const float* sAt, int Na, const uint8_t* Bt,
                       const float* sBt, int Nb, int ld, const int32_t* group_offsets, int G,
                       float* out0, float* out1, int split, int32_t* status, void* stream) {
    if (Na <= 0 || Nb <= 0 || G < 0 || ld < 0 || split <= 0 || split > Na) return MOE_ERR_INVALID_ARG;
    if (Na % 128 || Nb % 128 || split % 128 || ld % 16 || G > kMaxGroups) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((long long)G * Na > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (G == 0) return MOE_OK;
    if (!At || !sAt || !Bt || !sBt || !group_offsets || !out0 || (split < Na && !out1))
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(At) || !aligned16(Bt) || !aligned16(out0) || !aligned16(out1) ||
        !aligned16(sAt) || !aligned16(sBt))
        return MOE_ERR_MISALIGNED;
    return launch_wgrad_gemm(At, sAt, Na, Bt, sBt, Nb, ld, group_offsets, G, out0, out1, split,
                             status, S_(stream));
}

size_t moe_wgrad_workspace_size(const moe_layer_t* L, int T_max) {
    if (check_layer(L) || T_max < 0) return 0;
    const WgLayout W = wg_layout(T_max, L->d, L->E + L->S, L->K, L->S, L->I);
    return W.ld < 0 ? 0 : W.total;
}

int moe_backward_wgrad(const moe_layer_t* L, int T, float* dW_gate, float* dW_up, float* dW_down,
                       void* fwd_ws, size_t fwd_ws_bytes, void* bwd_ws, size_t bwd_ws_bytes,
                       void* wgrad_ws, size_t wgrad_ws_bytes, void* stream) {
    int rc = check_layer(L);
    if (rc) return rc;
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (!dW_gate || !dW_up || !dW_down || !fwd_ws || !bwd_ws || !wgrad_ws) return MOE_ERR_INVALID_ARG;
    if (!aligned16(dW_gate) || !aligned16(dW_up) || !aligned16(dW_down)) return MOE_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(fwd_ws) | reinterpret_cast<uintptr_t>(bwd_ws) |
         reinterpret_cast<uintptr_t>(wgrad_ws)) & 255u)
        return MOE_ERR_MISALIGNED;
    if ((long long)T * (L->K + L->S) > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int d = L->d, E = L->E, K = L->K, S = L->S, I = L->I, G = E + S;
    const Layout W = layout(T, d, E, K, S, I);
    const BwdLayout BW = bwd_layout(T, d, K, S, I);
    const WgLayout WG = wg_layout(T, d, G, K, S, I);
    if (WG.ld < 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (fwd_ws_bytes < W.total || bwd_ws_bytes < BW.total || wgrad_ws_bytes < WG.total)
        return MOE_ERR_WORKSPACE;
    const cudaStream_t st = S_(stream);
    if (T == 0) {                                    // no rows: every gradient is zero
        const size_t n = (size_t)G * I * d * sizeof(float);
        cudaError_t e = cudaMemsetAsync(dW_gate, 0, n, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(dW_up, 0, n, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(dW_down, 0, n, st);
        return e == cudaSuccess ? MOE_OK : cuda_fail(e);
    }
    char* fb = static_cast<char*>(fwd_ws);
    char* bb = static_cast<char*>(bwd_ws);
    char* wb = static_cast<char*>(wgrad_ws);
    int32_t* status = reinterpret_cast<int32_t*>(bb + BW.status);
    const int32_t* go = reinterpret_cast<const int32_t*>(fb + W.go);
    const int M = T * (K + S), ld = WG.ld;
    uint8_t* at = reinterpret_cast<uint8_t*>(wb + WG.at);
    uint8_t* ht = reinterpret_cast<uint8_t*>(wb + WG.ht);
    uint8_t* dyt = reinterpret_cast<uint8_t*>(wb + WG.dyt);
    uint8_t* gut = reinterpret_cast<uint8_t*>(wb + WG.gut);
    float* sat = reinterpret_cast<float*>(wb + WG.sat);
    float* sht = reinterpret_cast<float*>(wb + WG.sht);
    float* sdyt = reinterpret_cast<float*>(wb + WG.sdyt);
    float* sgut = reinterpret_cast<float*>(wb + WG.sgut);
    // the four held FP8 tensors in 128x1 tiles
    if ((rc = launch_requant_128x1(reinterpret_cast<const uint8_t*>(fb + W.A),
                                   reinterpret_cast<const float*>(fb + W.sa), M, d, go, G, at, sat, ld,
                                   status, st)))
        return rc;
    if ((rc = launch_requant_128x1(reinterpret_cast<const uint8_t*>(fb + W.H),
                                   reinterpret_cast<const float*>(fb + W.sh), M, I, go, G, ht, sht, ld,
                                   status, st)))
        return rc;
    if ((rc = launch_requant_128x1(reinterpret_cast<const uint8_t*>(bb + BW.dyq),
                                   reinterpret_cast<const float*>(bb + BW.sdy), M, d, go, G, dyt, sdyt,
                                   ld, status, st)))
        return rc;
    if ((rc = launch_requant_128x1(reinterpret_cast<const uint8_t*>(bb + BW.dgu),
                                   reinterpret_cast<const float*>(bb + BW.sgu), M, 2 * I, go, G, gut,
                                   sgut, ld, status, st)))
        return rc;
    // dW_down = dy^T h
    if ((rc = launch_wgrad_gemm(dyt, sdyt, d, ht, sht, I, ld, go, G, dW_down, nullptr, d, status, st)))
        return rc;
    // [dW_gate ; dW_up] = [dG | dU]^T A
    return launch_wgrad_gemm(gut, sgut, 2 * I, at, sat, d, ld, go, G, dW_gate, dW_up, I, status, st);
}

int moe_forward_host(const moe_layer_t* L, int T, int n_batches, const uint16_t* const* u_host,
                     float* const* h_host, float gamma, const moe_batch_buffers_t* buf, void* ws,
                     size_t ws_bytes, void* compute_stream, void* h2d_stream, void* d2h_stream) {
    int rc = check_layer(L);
    if (rc) return rc;
    if (T < 0 || n_batches < 0) return MOE_ERR_INVALID_ARG;
    if (n_batches == 0) return MOE_OK;
    if (!u_host || !h_host || !buf || !ws) return MOE_ERR_INVALID_ARG;
    for (int k = 0; k < n_batches; ++k)
        if (T > 0 && (!u_host[k] || !h_host[k])) return MOE_ERR_INVALID_ARG;
    for (int s = 0; s < 2; ++s) {
        const moe_batch_buffers_t& b = buf[s];
        if (!b.counts || (T > 0 && (!b.u || !b.h || !b.topk_idx || !b.topk_gate || !b.tie_flag)))
            return MOE_ERR_INVALID_ARG;
        if (!aligned16(b.u) || !aligned16(b.h)) return MOE_ERR_MISALIGNED;
    }
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_MISALIGNED;
    if (ws_bytes < layout(T, L->d, L->E, L->K, L->S, L->I).total) return MOE_ERR_WORKSPACE;
    const cudaStream_t cs = S_(compute_stream), up = S_(h2d_stream), down = S_(d2h_stream);
    EventSet E;
    cudaEvent_t* h2d_done = E.ev;          // [2] batch k's tokens are on the device
    cudaEvent_t* fwd_done = E.ev + 2;      // [2] batch k's forward (and bias step) finished
    cudaEvent_t* d2h_done = E.ev + 4;      // [2] batch k's output is in host memory
    cudaError_t e;
    for (cudaEvent_t& ev : E.ev)
        if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e);
    int32_t* status = static_cast<int32_t*>(ws);
    if ((e = cudaMemsetAsync(status, 0, 16, cs)) != cudaSuccess) return cuda_fail(e);
    const size_t u_bytes = sizeof(uint16_t) * (size_t)T * L->d;
    const size_t h_bytes = sizeof(float) * (size_t)T * L->d;
    for (int k = 0; k < n_batches; ++k) {
        const int s = k & 1;
        const moe_batch_buffers_t& b = buf[s];
        // upload into slot s once batch k-2's forward has read it
        if (k >= 2 && (e = cudaStreamWaitEvent(up, fwd_done[s], 0)) != cudaSuccess) return cuda_fail(e);
        if (T > 0 && (e = cudaMemcpyAsync(b.u, u_host[k], u_bytes, cudaMemcpyHostToDevice, up)) !=
                         cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaEventRecord(h2d_done[s], up)) != cudaSuccess) return cuda_fail(e);
        // forward once the tokens are there and slot s's output has been read back
        if ((e = cudaStreamWaitEvent(cs, h2d_done[s], 0)) != cudaSuccess) return cuda_fail(e);
        if (k >= 2 && (e = cudaStreamWaitEvent(cs, d2h_done[s], 0)) != cudaSuccess) return cuda_fail(e);
        if ((rc = forward_impl(L, b.u, T, b.h, b.topk_idx, b.topk_gate, b.counts, b.tie_flag, ws,
                               ws_bytes, cs, false)))
            return rc;
        if (gamma != 0.0f &&
            (rc = launch_update_bias(b.counts, L->E, T, L->K, gamma, const_cast<float*>(L->bias), cs)))
            return rc;
        if ((e = cudaEventRecord(fwd_done[s], cs)) != cudaSuccess) return cuda_fail(e);
        // download
        if ((e = cudaStreamWaitEvent(down, fwd_done[s], 0)) != cudaSuccess) return cuda_fail(e);
        if (T > 0 && (e = cudaMemcpyAsync(h_host[k], b.h, h_bytes, cudaMemcpyDeviceToHost, down)) !=
                         cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaEventRecord(d2h_done[s], down)) != cudaSuccess) return cuda_fail(e);
    }
    return MOE_OK;
}

int moe_forward_pipelined(const moe_layer_t* L, int T, int n_batches,
                          const moe_batch_buffers_t* batches, float gamma, void* ws0, void* ws1,
                          size_t ws_bytes, int reserve_sms, void* gemm_stream, void* side_stream) {
    int rc = check_layer(L);
    if (rc) return rc;
    if (T < 0 || n_batches < 0 || reserve_sms < 0) return MOE_ERR_INVALID_ARG;
    if (n_batches == 0) return MOE_OK;
    if (!batches) return MOE_ERR_INVALID_ARG;
    void* wss[2] = {ws0, ws1};
    for (int k = 0; k < n_batches; ++k) {
        const moe_batch_buffers_t& b = batches[k];
        if ((rc = check_forward(L, b.u, T, b.h, b.topk_idx, b.topk_gate, b.counts, b.tie_flag,
                                wss[k & 1], ws_bytes)))
            return rc;
    }
    int sms = 0, dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (reserve_sms >= sms) return MOE_ERR_INVALID_ARG;
    const int gemm_ctas = sms - reserve_sms;
    const cudaStream_t gs = S_(gemm_stream), ss = S_(side_stream);
    EventSet ev;
    cudaEvent_t* prep_done = ev.ev;        // [2] batch k's dispatch rows are ready
    cudaEvent_t* gemm_done = ev.ev + 2;    // [2] batch k's expert outputs are ready
    for (int i = 0; i < 4; ++i)
        if ((e = cudaEventCreateWithFlags(&ev.ev[i], cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e);
    Fwd f[2] = {fwd_ptrs(L, T, ws0), fwd_ptrs(L, T, ws1)};
    // side stream: prep(0), prep(1), combine(0), prep(2), combine(1), ... ; the
    // bias update of batch k sits between its routing and the next batch's, and
    // a workspace is reused by batch k + 2 only after batch k's combine
    auto combine = [&](int k) -> int {
        const moe_batch_buffers_t& b = batches[k];
        cudaError_t ce = cudaStreamWaitEvent(ss, gemm_done[k & 1], 0);
        if (ce != cudaSuccess) return cuda_fail(ce);
        return forward_combine(L, b.u, T, b.topk_gate, b.h, f[k & 1], ss);
    };
    for (int k = 0; k < n_batches; ++k) {
        const moe_batch_buffers_t& b = batches[k];
        const Fwd& fk = f[k & 1];
        if ((rc = forward_prep(L, b.u, T, b.topk_idx, b.topk_gate, b.counts, b.tie_flag, fk, ss,
                               k < 2)))
            return rc;
        if (gamma != 0.0f &&
            (rc = launch_update_bias(b.counts, L->E, T, L->K, gamma, const_cast<float*>(L->bias), ss)))
            return rc;
        if ((e = cudaEventRecord(prep_done[k & 1], ss)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaStreamWaitEvent(gs, prep_done[k & 1], 0)) != cudaSuccess) return cuda_fail(e);
        if ((rc = forward_gemms(L, T, fk, gs, gemm_ctas))) return rc;
        if ((e = cudaEventRecord(gemm_done[k & 1], gs)) != cudaSuccess) return cuda_fail(e);
        if (k >= 1 && (rc = combine(k - 1))) return rc;
    }
    return combine(n_batches - 1);
}

int moe_update_bias(const int32_t* counts, int E, int T, int K, float gamma, float* bias,
                    void* stream) {
    if (E <= 0 || T < 0 || K <= 0 || !counts || !bias) return MOE_ERR_INVALID_ARG;
    return launch_update_bias(counts, E, T, K, gamma, bias, S_(stream));
}

int moe_check_device_status(int32_t* status, void* stream) {
    if (!status) return MOE_ERR_INVALID_ARG;
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, status, sizeof(v), cudaMemcpyDeviceToHost, S_(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(S_(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    if (v != 0) {
        e = cudaMemsetAsync(status, 0, sizeof(int32_t), S_(stream));
        if (e == cudaSuccess) e = cudaStreamSynchronize(S_(stream));
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return v;
}

}  // extern "C"
