// Shared device helpers and internal launcher declarations of libmoefp8.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/moe_fp8.h"

namespace moe {

// Counts every kernel this library launches (reported by moe_kernel_launches).
void note_launch();
// Limit of the grouped GEMMs' pipeline waits in SM clock cycles
// (moe_set_pipeline_wait_limit; about 2 s by default).
long long pipeline_wait_cycles();
// Test switch of moe_set_pipeline_stall: the GEMM producers issue no loads.
int pipeline_stall();
// Records a failed CUDA call for moe_last_cuda_error and returns MOE_ERR_CUDA.
int cuda_fail(cudaError_t e);
// Checks the launch that was just made.
int check_launch();

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Two float32 -> two E4M3 codes, round to nearest even, saturating to +-448
// (the hardware conversion of sm_89+; `lo` ends up in the low byte).
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Quantise 4 values with one tile scale (IEEE division, as the scale rule).
__device__ __forceinline__ uint32_t quant4(float a, float b, float c, float d, float scale) {
    uint32_t lo = e4m3x2(__fdiv_rn(a, scale), __fdiv_rn(b, scale));
    uint32_t hi = e4m3x2(__fdiv_rn(c, scale), __fdiv_rn(d, scale));
    return lo | (hi << 16);
}

// Tile scale from the tile's max |x|: amax / 448, or 1 for an all-zero tile.
__device__ __forceinline__ float tile_scale(float amax) {
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

__device__ __forceinline__ void flag_status(int32_t* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// Programmatic dependent launch.  The kernels of the layer are launched with
// launch_pdl, so a kernel's CTAs can be scheduled while the previous kernel
// in the stream drains.  Every kernel therefore calls griddep_wait() before
// its first access to global memory (it returns once the previous kernel has
// completed and its writes are visible; without a programmatic predecessor
// it returns at once), then griddep_launch() so that the next kernel can be
// scheduled.  Correctness never depends on griddep_launch(): the next
// kernel's own griddep_wait() waits for this whole grid.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches `kernel` on `st` with programmatic stream serialization allowed
// (see griddep_wait); counts the launch and checks it.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
               Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    note_launch();
    return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

// ---------------------------------------------------------------- launchers
int launch_quant_1x128(const uint16_t* x, int n_src, const int32_t* gather, int n_gather,
                       int tail_T, int M, int d, uint8_t* q, float* scales, int scale_ld,
                       int32_t* status, cudaStream_t st);
int launch_quant_dispatch(const uint16_t* x, int T, int d, const int32_t* inv_row, int K, int S,
                          uint8_t* q, float* scales, int scale_ld, int32_t* status,
                          cudaStream_t st);
int launch_quant_128x128(const float* w, int R, int C, uint8_t* q, float* scales, cudaStream_t st);
// CUDA-core router (route.cu).  part (nullable): room for split-K partial
// logits (part_floats floats), summed in a fixed order; without it the
// partials are added atomically into logits.
int launch_route(const uint16_t* u, const float* cent, const float* bias, int T, int d, int E,
                 int K, int32_t* idx, float* gate, uint8_t* tie, int32_t* counts, float* logits,
                 cudaStream_t st, float* part = nullptr, size_t part_floats = 0);
// The tensor-core router of moe_route (route_tc.cu): workspace bytes for T
// tokens, and the launch (the workspace's first int32 is not touched; the
// status word is passed separately).
size_t route_ws_bytes(int T, int d, int E);
int launch_route_tc(const uint16_t* u, const float* cent, const float* bias, int T, int d, int E,
                    int K, int32_t* idx, float* gate, uint8_t* tie, int32_t* counts, void* ws,
                    int32_t* status, cudaStream_t st, int n_groups = 0, int topk_groups = 0,
                    int group_topk = 0);
// The layer's router: the CUDA-core exact router for small batches without
// group limits, else launch_route_tc (same workspace as launch_route_tc).
int launch_route_layer(const uint16_t* u, const float* cent, const float* bias, int T, int d, int E,
                       int K, int32_t* idx, float* gate, uint8_t* tie, int32_t* counts, void* ws,
                       int32_t* status, cudaStream_t st, int n_groups, int topk_groups,
                       int group_topk);
// The router's logit estimates summed into out [T, E], and the bound's
// centroid norms of the bound into norms_out [E] (device), for checking the bound.
int launch_route_estimate(const uint16_t* u, const float* cent, int T, int d, int E, float* out,
                          float* norms_out, void* ws, int32_t* status, cudaStream_t st);
// Input gradient of the layer (backward.cu, route_tc.cu).
int launch_transpose_blocks(const uint8_t* src, const float* ssrc, int G, int R, int C, uint8_t* dst,
                            int dst_ld, int col_off, float* sdst, int sdst_ld, int scol_off,
                            cudaStream_t st);
int launch_quant_dy(const uint16_t* dh, int T, int d, const float* gate, const int32_t* inv_row,
                    int K, int S, uint8_t* q, float* scales, int scale_ld, int32_t* status,
                    cudaStream_t st);
int launch_gate_term(const uint16_t* u, const uint16_t* dh, const uint16_t* Y, const int32_t* inv_row,
                     const int32_t* idx, const float* gate, const float* cent, int T, int d, int K,
                     int M, float* du, int32_t* status, cudaStream_t st);
// Weight gradients (wgrad.cu).
int launch_requant_128x1(const uint8_t* q, const float* s, int M, int C, const int32_t* go, int G,
                         uint8_t* qt, float* st, int ld, int32_t* status, cudaStream_t stream);
int launch_wgrad_gemm(const uint8_t* At, const float* sAt, int Na, const uint8_t* Bt,
                      const float* sBt, int Nb, int ld, const int32_t* go, int G, float* out0,
                      float* out1, int split, int32_t* status, cudaStream_t st);
int launch_permute(const int32_t* idx, int T, int K, int E, int32_t* offsets, int32_t* perm,
                   int32_t* inv_row, int32_t* group_offsets_ext, int S, int32_t* status,
                   int32_t* ws_hist, int32_t* ws_base, cudaStream_t st);
// DOWN modes: with out2 set, the rows of groups >= f32_group0 are stored as
// float32 in out2 (row - f32_row0) and the other rows as bf16 in out.  The
// tile counter is status[counter_slot], zeroed by the launcher unless
// counter_zeroed says the caller has.  max_ctas > 0 caps the persistent grid
// (the SMs left free run other work concurrently).
int launch_grouped_gemm(int mode, const uint8_t* A, const float* sa, int M_total,
                        const int32_t* go, int G, const uint8_t* W0, const uint8_t* W1,
                        const float* sw0, const float* sw1, int N, int Kdim, void* out,
                        float* out_scales, int32_t* status, cudaStream_t st,
                        const uint16_t* dH = nullptr, int f32_group0 = 1 << 30, int f32_row0 = 0,
                        float* out2 = nullptr, int counter_slot = 1, bool counter_zeroed = false,
                        int max_ctas = 0);
// The same GEMM with tiles of 128 weight rows x up to 32 rows of a group
// (gemm_small.cu; GATE_UP_SILU_QUANT and DOWN modes): for groups with few rows.
int launch_grouped_gemm_small(int mode, const uint8_t* A, const float* sa, int M_total,
                              const int32_t* go, int G, const uint8_t* W0, const uint8_t* W1,
                              const float* sw0, const float* sw1, int N, int Kdim, void* out,
                              float* out_scales, int32_t* status, cudaStream_t st,
                              int f32_group0 = 1 << 30, int f32_row0 = 0, float* out2 = nullptr,
                              int counter_slot = 1, bool counter_zeroed = false, int max_ctas = 0);
// The combine: routed rows Y bf16 with shared rows Ysh float32 (the forward),
// or both bf16 (the input gradient's rows, gathered with gate = NULL).
int launch_combine(const uint16_t* u, const uint16_t* Y, const float* gate, const int32_t* inv_row,
                   const uint16_t* Ysh, int T, int d, int K, int S, float* h, cudaStream_t st);
int launch_combine(const uint16_t* u, const uint16_t* Y, const float* gate, const int32_t* inv_row,
                   const float* Ysh, int T, int d, int K, int S, float* h, cudaStream_t st);
int launch_update_bias(const int32_t* counts, int E, int T, int K, float gamma, float* bias,
                       cudaStream_t st);

constexpr int kPermuteChunk = 64;   // tokens per block in the dispatch kernels
constexpr int kMaxGroups = 1088;    // E + S limit of the grouped GEMM
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace moe
