// Fine-grained FP8 quantisation kernels.
//
// Source: "รายงานเชิงเทคนิคของ DeepSeek-V3" (xyznot.com/th/paper/2412.19437),
// Key ideas, FP8 bullet (E4M3 everywhere; activations scaled per 1x128 tile,
// weights per 128x128 block) and "官方揭秘DeepSeek-V3模型训练全流程"
// (youleyou.com) §4.3 (the scale comes from the tile's max |x|, computed
// online).  Rule used here: scale = amax / 448, code = E4M3(x / scale) with
// round-to-nearest-even and saturation; an all-zero tile gets scale 1.
#include "common.cuh"

namespace moe {
namespace {

// One warp quantises one output row at a time; each lane owns 8 consecutive
// values (one 16-byte load), so a half-warp covers one 128-wide tile and a
// full warp two tiles.  Rows: [0, n_gather) take input row gather[r] (or r
// when gather is null); rows [n_gather, M) take input row (r - n_gather) %
// tail_T (the shared-expert copies of every token).
__global__ void __launch_bounds__(256) quant_1x128_kernel(
    const uint16_t* __restrict__ x, int n_src, const int32_t* __restrict__ gather, int n_gather,
    int tail_T, int M, int d, uint8_t* __restrict__ q, float* __restrict__ scales, int scale_ld,
    int32_t* status) {
    griddep_wait();
    griddep_launch();
    const int lane = threadIdx.x & 31;
    const int warps_per_block = blockDim.x >> 5;
    const int half = lane >> 4;          // which tile of the 256-wide step
    const int hl = lane & 15;            // lane within the tile
    for (int r = blockIdx.x * warps_per_block + (threadIdx.x >> 5); r < M;
         r += gridDim.x * warps_per_block) {
        int src;
        if (r < n_gather)
            src = gather ? gather[r] : r;
        else
            src = (r - n_gather) % tail_T;
        if (src < 0 || src >= n_src) {
            if (lane == 0) flag_status(status, MOE_ERR_BAD_INDEX);
            continue;
        }
        const uint16_t* xr = x + (size_t)src * d;
        uint8_t* qr = q + (size_t)r * d;
        for (int c0 = 0; c0 < d; c0 += 256) {
            const int col = c0 + half * 128 + hl * 8;
            const bool active = col < d;      // d % 256 == 128: upper half idle on the last step
            float v[8];
            float amax = 0.0f;
            if (active) {
                uint4 raw = *reinterpret_cast<const uint4*>(xr + col);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[2 * i] = bf16_bits_to_float(static_cast<uint16_t>(w[i] & 0xFFFFu));
                    v[2 * i + 1] = bf16_bits_to_float(static_cast<uint16_t>(w[i] >> 16));
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            if (active) {
                const float scale = tile_scale(amax);
                uint2 out;
                if (amax == 0.0f) {
                    out = make_uint2(0u, 0u);
                } else {
                    out.x = quant4(v[0], v[1], v[2], v[3], scale);
                    out.y = quant4(v[4], v[5], v[6], v[7], scale);
                }
                *reinterpret_cast<uint2*>(qr + col) = out;
                if (hl == 0) scales[(size_t)(col >> 7) * scale_ld + r] = scale;
            }
        }
    }
}

// Quantise every token once and write its codes to all the rows the
// dispatch gave it: routed rows inv_row[t, 0..K) and shared rows
// T*K + s*T + t.  One warp per work item; each lane owns 8 consecutive values
// of a 256-wide step (a half-warp per 128-wide tile), exactly as
// quant_1x128_kernel, so codes and scales are the same bits.  A work item is
// SUB consecutive 256-wide steps of one token: the lanes issue all SUB loads
// before any reduction, so a warp has SUB x 512 bytes of the token in flight
// (SUB = 4 for large batches; 1 when there are few tokens, to spread them
// over more warps).
template <int SUB>
__global__ void __launch_bounds__(256) quant_dispatch_kernel(
    const uint16_t* __restrict__ x, int T, int d, const int32_t* __restrict__ inv_row, int K,
    int S, int M, uint8_t* __restrict__ q, float* __restrict__ scales, int scale_ld,
    int32_t* status) {
    griddep_wait();
    griddep_launch();
    const int lane = threadIdx.x & 31;
    const int warps_per_block = blockDim.x >> 5;
    const int half = lane >> 4;
    const int hl = lane & 15;
    const int nch = (d + 256 * SUB - 1) / (256 * SUB);
    const long long items = (long long)T * nch;
    for (long long item = (long long)blockIdx.x * warps_per_block + (threadIdx.x >> 5); item < items;
         item += (long long)gridDim.x * warps_per_block) {
        const int t = (int)(item / nch);
        const int c0 = (int)(item % nch) * 256 * SUB;
        // lane j < K holds routed row j of this token, lane K + s shared row s
        int my_row = -1;
        if (lane < K) {
            my_row = inv_row[(size_t)t * K + lane];
            if (my_row < 0 || my_row >= M) {
                flag_status(status, MOE_ERR_BAD_INDEX);
                my_row = -1;
            }
        } else if (lane < K + S) {
            my_row = T * K + (lane - K) * T + t;
        }
        const int R = K + S;
        const uint16_t* xr = x + (size_t)t * d;
        uint4 raw[SUB];
#pragma unroll
        for (int j = 0; j < SUB; ++j) {
            const int col = c0 + j * 256 + half * 128 + hl * 8;
            raw[j] = col < d ? *reinterpret_cast<const uint4*>(xr + col) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < SUB; ++j) {
            const int col = c0 + j * 256 + half * 128 + hl * 8;
            if (c0 + j * 256 >= d) break;                 // warp-uniform
            const bool active = col < d;
            float v[8];
            float amax = 0.0f;
            const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[2 * i] = bf16_bits_to_float(static_cast<uint16_t>(w[i] & 0xFFFFu));
                v[2 * i + 1] = bf16_bits_to_float(static_cast<uint16_t>(w[i] >> 16));
            }
            if (active) {
#pragma unroll
                for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            const float scale = tile_scale(amax);
            uint2 out = make_uint2(0u, 0u);
            if (active && amax != 0.0f) {
                out.x = quant4(v[0], v[1], v[2], v[3], scale);
                out.y = quant4(v[4], v[5], v[6], v[7], scale);
            }
            for (int r = 0; r < R; ++r) {
                const int row = __shfl_sync(0xffffffffu, my_row, r);
                if (row < 0) continue;
                if (active) {
                    *reinterpret_cast<uint2*>(q + (size_t)row * d + col) = out;
                    if (hl == 0) scales[(size_t)(col >> 7) * scale_ld + row] = scale;
                }
            }
        }
    }
}

// One block quantises one 128x128 weight block: 256 threads, 64 values each.
__global__ void __launch_bounds__(256) quant_128x128_kernel(const float* __restrict__ w, int R,
                                                            int C, uint8_t* __restrict__ q,
                                                            float* __restrict__ scales) {
    const int bc = blockIdx.x, br = blockIdx.y;
    const int tid = threadIdx.x;
    // Value e = i * 1024 + tid * 4 (+0..3) of the row-major 128x128 block, i = 0..15:
    // every load instruction of a warp covers 512 contiguous bytes of one row group.
    float4 v[16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int e = i * 1024 + tid * 4;
        const int r = e >> 7, c = e & 127;
        v[i] = *reinterpret_cast<const float4*>(w + (size_t)(br * 128 + r) * C + bc * 128 + c);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)),
                                 fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
    }
    __shared__ float red[8];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    const float scale = tile_scale(amax);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int e = i * 1024 + tid * 4;
        const int r = e >> 7, c = e & 127;
        const uint32_t code = amax == 0.0f ? 0u : quant4(v[i].x, v[i].y, v[i].z, v[i].w, scale);
        *reinterpret_cast<uint32_t*>(q + (size_t)(br * 128 + r) * C + bc * 128 + c) = code;
    }
    if (tid == 0) scales[(size_t)br * (C / 128) + bc] = scale;
}

}  // namespace

int launch_quant_1x128(const uint16_t* x, int n_src, const int32_t* gather, int n_gather,
                       int tail_T, int M, int d, uint8_t* q, float* scales, int scale_ld,
                       int32_t* status, cudaStream_t st) {
    if (M == 0) return MOE_OK;
    const int warps = 8;
    int blocks = (M + warps - 1) / warps;
    if (blocks > 148 * 16) blocks = 148 * 16;
    return launch_pdl(quant_1x128_kernel, dim3(blocks), dim3(warps * 32), 0, st, x, n_src, gather,
                      n_gather, tail_T > 0 ? tail_T : 1, M, d, q, scales, scale_ld, status);
}

int launch_quant_dispatch(const uint16_t* x, int T, int d, const int32_t* inv_row, int K, int S,
                          uint8_t* q, float* scales, int scale_ld, int32_t* status,
                          cudaStream_t st) {
    if (T == 0) return MOE_OK;
    const int warps = 8;
    // four 256-wide steps per work item once there are enough items for every
    // resident warp (148 SMs x 64 warps)
    const long long items1 = (long long)T * ((d + 255) / 256);
    const bool wide = items1 >= 4LL * 148 * 64;
    const long long items = wide ? (long long)T * ((d + 1023) / 1024) : items1;
    const int blocks = (int)((items + warps - 1) / warps < 148 * 16 ? (items + warps - 1) / warps : 148 * 16);
    if (wide)
        return launch_pdl(quant_dispatch_kernel<4>, dim3(blocks), dim3(warps * 32), 0, st, x, T, d,
                          inv_row, K, S, T * (K + S), q, scales, scale_ld, status);
    return launch_pdl(quant_dispatch_kernel<1>, dim3(blocks), dim3(warps * 32), 0, st, x, T, d, inv_row,
                      K, S, T * (K + S), q, scales, scale_ld, status);
}

int launch_quant_128x128(const float* w, int R, int C, uint8_t* q, float* scales,
                         cudaStream_t st) {
    if (R == 0 || C == 0) return MOE_OK;
    dim3 grid(C / 128, R / 128);
    quant_128x128_kernel<<<grid, 256, 0, st>>>(w, R, C, q, scales);
    return check_launch();
}

}  // namespace moe
