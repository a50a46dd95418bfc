// Input gradient of the layer: the pieces that are not the grouped GEMM.
//
// The pages say only that FP8 carries the inputs and part of the gradient
// propagation ("DeepSeek V3技術報告", FP8 資料格式訓練) and ask for
// transposed-GEMM support in hardware ("官方揭秘DeepSeek-V3模型训练全流程",
// hardware suggestions).  Reading: the backward GEMMs follow the forward's FP8
// rule.  A weight's transpose is exact in FP8 with 128x128 block scales: the
// codes move, each block keeps its scale.  The expert-output gradient of a
// routed row is g_k * dh (a float32 product) and of a shared row dh, each
// quantised per 1x128 tile with the forward's rule.
#include "common.cuh"

namespace moe {
namespace {

// One 128x128 block of W [R, C] (group g) to W^T: dst[g][c][col_off + r] in
// rows of dst_ld codes, and its scale to sdst[g][c / 128][scol_off + r / 128]
// in rows of sdst_ld.
__global__ void __launch_bounds__(256) transpose_blocks_kernel(
    const uint8_t* __restrict__ src, const float* __restrict__ ssrc, int R, int C,
    uint8_t* __restrict__ dst, int dst_ld, int col_off, float* __restrict__ sdst, int sdst_ld,
    int scol_off) {
    __shared__ uint8_t tile[128][128 + 16];
    const int nbc = C / 128, nbr = R / 128;
    const int g = blockIdx.z, bi = blockIdx.y, bj = blockIdx.x;
    const uint8_t* s = src + ((size_t)g * R + (size_t)bi * 128) * C + (size_t)bj * 128;
    for (int i = threadIdx.x; i < 128 * 8; i += 256) {
        const int r = i >> 3, q = i & 7;
        *reinterpret_cast<uint4*>(&tile[r][q * 16]) =
            *reinterpret_cast<const uint4*>(s + (size_t)r * C + q * 16);
    }
    __syncthreads();
    // output row c (of the transposed block), 128 codes from column c of the tile
    uint8_t* d = dst + ((size_t)g * C + (size_t)bj * 128) * dst_ld + col_off + (size_t)bi * 128;
    for (int i = threadIdx.x; i < 128 * 8; i += 256) {
        const int c = i >> 3, q = i & 7;
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int r = q * 16 + k * 4;
            w[k] = (uint32_t)tile[r][c] | ((uint32_t)tile[r + 1][c] << 8) |
                   ((uint32_t)tile[r + 2][c] << 16) | ((uint32_t)tile[r + 3][c] << 24);
        }
        *reinterpret_cast<uint4*>(d + (size_t)c * dst_ld + q * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (threadIdx.x == 0)
        sdst[((size_t)g * nbc + bj) * sdst_ld + scol_off + bi] = ssrc[((size_t)g * nbr + bi) * nbc + bj];
}

// One warp per token: every dispatch row of the token gets its gradient
// (g_k dh for routed slot k, dh for a shared expert) quantised per 1x128
// tile.  Lane L holds elements 4L .. 4L + 3 of each tile.
__global__ void __launch_bounds__(256) quant_dy_kernel(const uint16_t* __restrict__ dh, int T, int d,
                                                      const float* __restrict__ gate,
                                                      const int32_t* __restrict__ inv_row, int K,
                                                      int S, uint8_t* __restrict__ q,
                                                      float* __restrict__ scales, int scale_ld,
                                                      int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const int M = T * (K + S);
    for (int r = 0; r < K + S; ++r) {
        const bool routed = r < K;
        const int row = routed ? inv_row[(size_t)t * K + r] : T * K + (r - K) * T + t;
        if (row < 0 || row >= M) {
            if (lane == 0) flag_status(status, MOE_ERR_BAD_INDEX);
            continue;
        }
        const float gk = routed ? gate[(size_t)t * K + r] : 1.0f;
        for (int kb = 0; kb < d / 128; ++kb) {
            const uint2 v = *reinterpret_cast<const uint2*>(dh + (size_t)t * d + kb * 128 + lane * 4);
            float x[4] = {bf16_bits_to_float(static_cast<uint16_t>(v.x & 0xFFFFu)),
                          bf16_bits_to_float(static_cast<uint16_t>(v.x >> 16)),
                          bf16_bits_to_float(static_cast<uint16_t>(v.y & 0xFFFFu)),
                          bf16_bits_to_float(static_cast<uint16_t>(v.y >> 16))};
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (routed) x[i] = gk * x[i];
                amax = fmaxf(amax, fabsf(x[i]));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            const float scale = tile_scale(amax);
            const uint32_t codes = amax == 0.0f ? 0u : quant4(x[0], x[1], x[2], x[3], scale);
            *reinterpret_cast<uint32_t*>(q + (size_t)row * d + kb * 128 + lane * 4) = codes;
            if (lane == 0) scales[(size_t)kb * scale_ld + row] = scale;
        }
    }
}

}  // namespace

int launch_transpose_blocks(const uint8_t* src, const float* ssrc, int G, int R, int C, uint8_t* dst,
                            int dst_ld, int col_off, float* sdst, int sdst_ld, int scol_off,
                            cudaStream_t st) {
    if (G == 0 || R == 0 || C == 0) return MOE_OK;
    transpose_blocks_kernel<<<dim3(C / 128, R / 128, G), 256, 0, st>>>(src, ssrc, R, C, dst, dst_ld,
                                                                      col_off, sdst, sdst_ld, scol_off);
    return check_launch();
}

int launch_quant_dy(const uint16_t* dh, int T, int d, const float* gate, const int32_t* inv_row,
                    int K, int S, uint8_t* q, float* scales, int scale_ld, int32_t* status,
                    cudaStream_t st) {
    if (T == 0) return MOE_OK;
    quant_dy_kernel<<<(T + 7) / 8, 256, 0, st>>>(dh, T, d, gate, inv_row, K, S, q, scales, scale_ld,
                                                 status);
    return check_launch();
}

}  // namespace moe
