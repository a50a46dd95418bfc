// Layer output and bias update.
//
// Source: "รายงานเชิงเทคนิคของ DeepSeek-V3" (xyznot.com/th/paper/2412.19437),
// Method §2: h'_t = u_t + sum_{i <= N_s} FFN_i^(s)(u_t) + sum_{i <= N_r}
// g_{i,t} FFN_i^(r)(u_t); and the end-of-step rule b_i <- b_i - gamma for an
// overloaded expert, b_i <- b_i + gamma for an underloaded one.
#include "common.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], uint4 raw, float w) {
    const uint32_t v[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(w, bf16_bits_to_float(static_cast<uint16_t>(v[i] & 0xFFFFu)), acc[2 * i]);
        acc[2 * i + 1] = fmaf(w, bf16_bits_to_float(static_cast<uint16_t>(v[i] >> 16)), acc[2 * i + 1]);
    }
}

__device__ __forceinline__ void add_f32x8(float (&acc)[8], const float* src, float w) {
    const float4 a = *reinterpret_cast<const float4*>(src);
    const float4 b = *reinterpret_cast<const float4*>(src + 4);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = fmaf(w, v[i], acc[i]);
}
__device__ __forceinline__ void add_row8(float (&acc)[8], const uint16_t* src, float w) {
    add_bf16x8(acc, *reinterpret_cast<const uint4*>(src), w);
}
__device__ __forceinline__ void add_row8(float (&acc)[8], const float* src, float w) {
    add_f32x8(acc, src, w);
}

// One work item = one token's chunk of 8 * blockDim columns (grid-stride), so
// a few tokens still spread over many blocks; each thread owns 8 consecutive
// columns.  Sum order: u, shared experts, routed experts by slot.  gate NULL:
// every routed row has weight 1 (the input gradient's gather).  Routed rows Y
// are bf16 bits; shared rows Ysh float (the forward keeps the shared experts'
// outputs in float32) or bf16 bits (the gradient rows).
template <typename YST>
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ u,
                                                      const uint16_t* __restrict__ Y,
                                                      const float* __restrict__ gate,
                                                      const int32_t* __restrict__ inv_row,
                                                      const YST* __restrict__ Ysh, int T,
                                                      int d, int K, int S,
                                                      float* __restrict__ h) {
    __shared__ int rows[kMaxTopK];
    __shared__ float gs[kMaxTopK];
    griddep_wait();
    griddep_launch();
    const int chunk = blockDim.x * 8;
    const int nch = (d + chunk - 1) / chunk;
    const long long items = (long long)T * nch;
    for (long long item = blockIdx.x; item < items; item += gridDim.x) {
        const int t = (int)(item / nch);
        __syncthreads();
        if (threadIdx.x < K) {
            rows[threadIdx.x] = inv_row[(size_t)t * K + threadIdx.x];
            gs[threadIdx.x] = gate ? gate[(size_t)t * K + threadIdx.x] : 1.0f;
        }
        __syncthreads();
        {
            const int c = (int)(item % nch) * chunk + threadIdx.x * 8;
            if (c >= d) continue;
            float acc[8];
            const uint4 ur = *reinterpret_cast<const uint4*>(u + (size_t)t * d + c);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
            add_bf16x8(acc, ur, 1.0f);
            for (int s = 0; s < S; ++s) add_row8(acc, Ysh + ((size_t)s * T + t) * d + c, 1.0f);
            for (int k = 0; k < K; ++k) add_row8(acc, Y + (size_t)rows[k] * d + c, gs[k]);
            float4* out = reinterpret_cast<float4*>(h + (size_t)t * d + c);
            out[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            out[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
    }
}

__global__ void update_bias_kernel(const int32_t* __restrict__ counts, int E, long long n,
                                   float gamma, float* __restrict__ bias) {
    griddep_wait();
    griddep_launch();
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x) {
        const long long load = (long long)counts[e] * E;
        if (load > n)
            bias[e] = bias[e] - gamma;
        else if (load < n)
            bias[e] = bias[e] + gamma;
    }
}

}  // namespace

template <typename YST>
int launch_combine_t(const uint16_t* u, const uint16_t* Y, const float* gate, const int32_t* inv_row,
                     const YST* Ysh, int T, int d, int K, int S, float* h, cudaStream_t st) {
    if (T == 0) return MOE_OK;
    const int threads = 128;
    const long long items = (long long)T * ((d + threads * 8 - 1) / (threads * 8));
    const int blocks = (int)(items < 148 * 16 ? items : 148 * 16);
    return launch_pdl(combine_kernel<YST>, dim3(blocks), dim3(threads), 0, st, u, Y, gate, inv_row,
                      Ysh, T, d, K, S, h);
}

int launch_combine(const uint16_t* u, const uint16_t* Y, const float* gate, const int32_t* inv_row,
                   const uint16_t* Ysh, int T, int d, int K, int S, float* h, cudaStream_t st) {
    return launch_combine_t(u, Y, gate, inv_row, Ysh, T, d, K, S, h, st);
}

int launch_combine(const uint16_t* u, const uint16_t* Y, const float* gate, const int32_t* inv_row,
                   const float* Ysh, int T, int d, int K, int S, float* h, cudaStream_t st) {
    return launch_combine_t(u, Y, gate, inv_row, Ysh, T, d, K, S, h, st);
}

int launch_update_bias(const int32_t* counts, int E, int T, int K, float gamma, float* bias,
                       cudaStream_t st) {
    return launch_pdl(update_bias_kernel, dim3((E + 255) / 256), dim3(256), 0, st, counts, E,
                      (long long)T * K, gamma, bias);
}

}  // namespace moe
