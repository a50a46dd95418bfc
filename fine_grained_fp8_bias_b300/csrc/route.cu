// Router: affinity logits, sigmoid, bias-steered top-K, gate normalisation.
//
// Source: "รายงานเชิงเทคนิคของ DeepSeek-V3" (xyznot.com/th/paper/2412.19437),
// Method §2: s_{i,t} = Sigmoid(u_t^T e_i); g'_{i,t} = s_{i,t} when
// s_{i,t} + b_i is among the top K_r of {s_{j,t} + b_j}, else 0; g is g'
// normalised.  "Deepseek V3 国货之光 开源之光" (databean.com.cn), section
// "Auxiliary-Loss-Free Load Balancing": the bias b_i only steers which
// experts are chosen; the gate values use the unbiased s.
//
// Two kernels: the logits l = u E^T on CUDA cores (a tiled float32 GEMM, or
// for at most kSmallT tokens one block per expert streaming its centroid
// row), then one warp per token for sigmoid, selection and gates.  Used by
// moe_route_noalloc and, below 256 tokens, by the layer.  The logits feed a
// selection whose near-tie band is 1e-6 wide, so they are summed with
// compensation: each 32-element chunk is a plain FMA chain, and the chunk
// sums are added with TwoSum (Knuth's error-free addition), keeping the
// logit error near one float32 rounding instead of growing with d.
// Selection order: descending s + b, equal scores broken by the lower expert
// index.  Near-tie flag: the K-th and (K+1)-th biased scores differ by less
// than 1e-6.
#include <cfloat>
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr int LT = 64;   // tokens per logits tile
constexpr int LE = 64;   // experts per logits tile
constexpr int LK = 32;   // d per smem step

// Error-free sum (Knuth's TwoSum): s + err == a + b exactly.
__device__ __forceinline__ float two_sum(float a, float b, float& err) {
    const float s = a + b;
    const float bb = s - a;
    err = (a - (s - bb)) + (b - bb);
    return s;
}

// l[t, e] (+)= sum_{j in this block's d-range} u[t, j] * c[e, j].
// 256 threads, each computing a 4 x 4 patch of the 64 x 64 tile.  Every
// 32-term chunk of a dot product is a plain FMA chain started from zero;
// the chunk is then added into the running sum with TwoSum, and the
// rounding errors are kept in a separate compensation term (so only the
// short chains round inexactly).  With split > 1 (few tokens) every block
// writes its partial sum to part[split index][t][e] (the selection kernel adds
// them in a fixed order), or, without a partial buffer, adds it atomically
// into a zeroed l (the sum's last bits then depend on the arrival order).
__global__ void __launch_bounds__(256) logits_kernel(const uint16_t* __restrict__ u,
                                                     const float* __restrict__ c, int T, int d,
                                                     int E, int split, float* __restrict__ l,
                                                     float* __restrict__ part,
                                                     int32_t* __restrict__ counts) {
    __shared__ __align__(16) float us[LK][LT];
    __shared__ __align__(16) float cs[LK][LE];
    griddep_wait();
    griddep_launch();
    const int tid = threadIdx.x;
    // the selection kernel that follows adds into counts
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
        for (int e = tid; e < E; e += blockDim.x) counts[e] = 0;
    const int t0 = blockIdx.x * LT, e0 = blockIdx.y * LE;
    const int steps = d / LK;
    const int s_begin = (int)((long long)steps * blockIdx.z / split);
    const int s_end = (int)((long long)steps * (blockIdx.z + 1) / split);
    const int ty = tid >> 4, tx = tid & 15;
    float acc[4][4], cmp[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = cmp[i][j] = 0.0f;
    // loader mapping: a warp covers 32 consecutive rows at the same k offset,
    // so the transposed shared-memory stores hit 32 different banks.  The next
    // step's tile is fetched into registers while the current one is used.
    const int lrow = tid & 63;
    const int lk = (tid >> 6) * 8;
    const bool t_ok = t0 + lrow < T, e_ok = e0 + lrow < E;
    const uint16_t* urow = u + (size_t)(t_ok ? t0 + lrow : 0) * d + lk;
    const float* crow = c + (size_t)(e_ok ? e0 + lrow : 0) * d + lk;
    uint4 ureg = make_uint4(0u, 0u, 0u, 0u);
    float4 ca = make_float4(0.f, 0.f, 0.f, 0.f), cb = ca;
    auto fetch = [&](int step) {
        const int k0 = step * LK;
        if (t_ok) ureg = *reinterpret_cast<const uint4*>(urow + k0);
        if (e_ok) {
            ca = *reinterpret_cast<const float4*>(crow + k0);
            cb = *reinterpret_cast<const float4*>(crow + k0 + 4);
        }
    };
    if (s_begin < s_end) fetch(s_begin);
    for (int s = s_begin; s < s_end; ++s) {
        {
            const uint32_t w[4] = {ureg.x, ureg.y, ureg.z, ureg.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                us[lk + 2 * i][lrow] = bf16_bits_to_float(static_cast<uint16_t>(w[i] & 0xFFFFu));
                us[lk + 2 * i + 1][lrow] = bf16_bits_to_float(static_cast<uint16_t>(w[i] >> 16));
            }
            cs[lk + 0][lrow] = ca.x; cs[lk + 1][lrow] = ca.y; cs[lk + 2][lrow] = ca.z; cs[lk + 3][lrow] = ca.w;
            cs[lk + 4][lrow] = cb.x; cs[lk + 5][lrow] = cb.y; cs[lk + 6][lrow] = cb.z; cs[lk + 7][lrow] = cb.w;
        }
        __syncthreads();
        if (s + 1 < s_end) fetch(s + 1);
        float part[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) part[i][j] = 0.0f;
#pragma unroll
        for (int k = 0; k < LK; ++k) {
            const float4 a = *reinterpret_cast<const float4*>(&us[k][ty * 4]);
            const float4 b = *reinterpret_cast<const float4*>(&cs[k][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) part[i][j] = fmaf(av[i], bv[j], part[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float err;
                acc[i][j] = two_sum(acc[i][j], part[i][j], err);
                cmp[i][j] += err;
            }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx * 4 + j;
            if (e >= E) continue;
            const float v = acc[i][j] + cmp[i][j];
            if (split == 1)
                l[(size_t)t * E + e] = v;
            else if (part)
                part[((size_t)blockIdx.z * T + t) * E + e] = v;
            else
                atomicAdd(&l[(size_t)t * E + e], v);
        }
    }
}

// Few tokens (T <= kSmallT): one block of four warps per expert computes that
// expert's logit for every token, streaming the centroid row once with its
// loads spread over the four warps.  Warp w takes the 128-column chunks
// w, w + 4, ...; lane L holds columns 4 L .. 4 L + 3 of each chunk.  Each run
// of up to eight of a warp's chunks (32 products per lane and token) is a plain
// FMA chain, added with TwoSum; the lanes' sums are combined by a TwoSum
// butterfly, and the four warps' sums in warp order by thread 0.  No split
// partials, no atomics: the result does not depend on timing.
constexpr int kSmallT = 8;
__global__ void __launch_bounds__(128) logits_small_kernel(const uint16_t* __restrict__ u,
                                                           const float* __restrict__ c, int T,
                                                           int d, int E, float* __restrict__ l,
                                                           int32_t* __restrict__ counts) {
    __shared__ float wacc[4][kSmallT], wcmp[4][kSmallT];
    griddep_wait();
    griddep_launch();
    const int e = blockIdx.x;
    if (threadIdx.x == 0) counts[e] = 0;        // the selection kernel that follows adds into counts
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float* crow = c + (size_t)e * d + lane * 4;
    float acc[kSmallT], cmp[kSmallT], chain[kSmallT];
#pragma unroll
    for (int t = 0; t < kSmallT; ++t) acc[t] = cmp[t] = chain[t] = 0.0f;
    const int nch = d / 128;
    for (int c0 = warp; c0 < nch; c0 += 32) {           // eight of this warp's chunks per pass
        float4 cv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (c0 + 4 * i < nch) cv[i] = *reinterpret_cast<const float4*>(crow + (size_t)(c0 + 4 * i) * 128);
#pragma unroll
        for (int t = 0; t < kSmallT; ++t) {
            if (t >= T) break;
            const uint16_t* ur = u + (size_t)t * d + lane * 4;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (c0 + 4 * i >= nch) break;
                const uint2 w = *reinterpret_cast<const uint2*>(ur + (size_t)(c0 + 4 * i) * 128);
                chain[t] = fmaf(bf16_bits_to_float(static_cast<uint16_t>(w.x & 0xFFFFu)), cv[i].x, chain[t]);
                chain[t] = fmaf(bf16_bits_to_float(static_cast<uint16_t>(w.x >> 16)), cv[i].y, chain[t]);
                chain[t] = fmaf(bf16_bits_to_float(static_cast<uint16_t>(w.y & 0xFFFFu)), cv[i].z, chain[t]);
                chain[t] = fmaf(bf16_bits_to_float(static_cast<uint16_t>(w.y >> 16)), cv[i].w, chain[t]);
            }
            float err;
            acc[t] = two_sum(acc[t], chain[t], err);
            cmp[t] += err;
            chain[t] = 0.0f;
        }
    }
#pragma unroll
    for (int t = 0; t < kSmallT; ++t) {
        if (t >= T) break;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float oa = __shfl_xor_sync(0xffffffffu, acc[t], off);
            const float oc = __shfl_xor_sync(0xffffffffu, cmp[t], off);
            float err;
            acc[t] = two_sum(acc[t], oa, err);
            cmp[t] = (cmp[t] + oc) + err;
        }
        if (lane == 0) {
            wacc[warp][t] = acc[t];
            wcmp[warp][t] = cmp[t];
        }
    }
    __syncthreads();
    if (threadIdx.x < T) {
        const int t = threadIdx.x;
        float a = wacc[0][t], cm = wcmp[0][t];
#pragma unroll
        for (int w = 1; w < 4; ++w) {
            float err;
            a = two_sum(a, wacc[w][t], err);
            cm = (cm + wcmp[w][t]) + err;
        }
        l[(size_t)t * E + e] = a + cm;
    }
}

// Larger score first; equal scores: lower expert index first.
__device__ __forceinline__ bool better(float za, int ia, float zb, int ib) {
    return za > zb || (za == zb && ia < ib);
}

// One warp per token.  Lane L holds experts L, L + 32, ... (NV per lane).
// With part != NULL the logit is the sum of the split partials, added in
// split order with TwoSum compensation.
template <int NV>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ l,
                                                   const float* __restrict__ part, int split,
                                                   const float* __restrict__ bias, int T, int E,
                                                   int K, int32_t* __restrict__ idx,
                                                   float* __restrict__ gate,
                                                   uint8_t* __restrict__ tie,
                                                   int32_t* __restrict__ counts) {
    griddep_wait();
    griddep_launch();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    float s[NV], z[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const int e = j * 32 + lane;
        if (e < E) {
            float x;
            if (part) {
                // eight partials loaded at a time, then added in split order
                float acc = 0.0f, cmp = 0.0f;
                for (int z0 = 0; z0 < split; z0 += 8) {
                    float v[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        v[i] = z0 + i < split ? part[((size_t)(z0 + i) * T + t) * E + e] : 0.0f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (z0 + i >= split) break;
                        float err;
                        acc = two_sum(acc, v[i], err);
                        cmp += err;
                    }
                }
                x = acc + cmp;
            } else {
                x = l[(size_t)t * E + e];
            }
            s[j] = __fdiv_rn(1.0f, 1.0f + expf(-x));
            z[j] = s[j] + bias[e];
        } else {
            s[j] = 0.0f;
            z[j] = -FLT_MAX;
        }
    }
    unsigned taken = 0;                 // bit j: my expert j*32+lane already selected
    float my_s = 0.0f, ssum = 0.0f, zk = 0.0f, zk1 = 0.0f;
    int my_e = -1;
    const int rounds = K < E ? K + 1 : K;
    for (int k = 0; k < rounds; ++k) {
        float bz = -FLT_MAX;
        int be = 0x7fffffff, bj = -1;
        float bs = 0.0f;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int e = j * 32 + lane;
            if (e < E && !(taken >> j & 1u) && better(z[j], e, bz, be)) {
                bz = z[j]; be = e; bj = j; bs = s[j];
            }
        }
        float wz = bz, ws = bs;
        int we = be;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float oz = __shfl_xor_sync(0xffffffffu, wz, off);
            const int oe = __shfl_xor_sync(0xffffffffu, we, off);
            const float os = __shfl_xor_sync(0xffffffffu, ws, off);
            if (better(oz, oe, wz, we)) { wz = oz; we = oe; ws = os; }
        }
        if (we == be && bj >= 0) taken |= 1u << bj;     // the owner marks it
        if (k < K) {
            ssum += ws;                                  // same order in every lane
            if (lane == k) { my_e = we; my_s = ws; }
            if (k == K - 1) zk = wz;
        } else {
            zk1 = wz;
        }
    }
    if (lane < K) {
        idx[(size_t)t * K + lane] = my_e;
        gate[(size_t)t * K + lane] = __fdiv_rn(my_s, ssum);
        atomicAdd(&counts[my_e], 1);
    }
    if (lane == 0) tie[t] = (K < E && (zk - zk1) < 1e-6f) ? 1 : 0;
}

template <int NV>
int launch_topk_nv(const float* l, const float* part, int split, const float* bias, int T, int E,
                   int K, int32_t* idx, float* gate, uint8_t* tie, int32_t* counts,
                   cudaStream_t st) {
    const int warps = 8;
    return launch_pdl(topk_kernel<NV>, dim3((T + warps - 1) / warps), dim3(warps * 32), 0, st, l,
                      part, split, bias, T, E, K, idx, gate, tie, counts);
}

}  // namespace

int launch_route(const uint16_t* u, const float* cent, const float* bias, int T, int d, int E,
                 int K, int32_t* idx, float* gate, uint8_t* tie, int32_t* counts, float* logits,
                 cudaStream_t st, float* part, size_t part_floats) {
    cudaError_t e;
    if (T == 0) {
        e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)E, st);
        return e == cudaSuccess ? MOE_OK : cuda_fail(e);
    }
    int rc;
    const int gx = (T + LT - 1) / LT, gy = (E + LE - 1) / LE;
    int split = 1;
    if (T <= kSmallT) {
        if ((rc = launch_pdl(logits_small_kernel, dim3(E), dim3(128), 0, st, u, cent, T, d, E, logits,
                             counts)))
            return rc;
        part = nullptr;
    } else {
        const int target = 2 * 148;
        while (gx * gy * split < target && split * 2 <= d / LK / 4) split *= 2;
        // with a partial buffer, as many splits as it holds (a fixed summation order)
        if (part)
            while (split > 1 && (size_t)split * T * E > part_floats) split /= 2;
        const bool use_part = part && split > 1;
        if (split > 1 && !use_part) {
            e = cudaMemsetAsync(logits, 0, sizeof(float) * (size_t)T * E, st);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        if ((rc = launch_pdl(logits_kernel, dim3(gx, gy, split), dim3(256), 0, st, u, cent, T, d, E,
                             split, logits, use_part ? part : nullptr, counts)))
            return rc;
        if (!use_part) part = nullptr;
    }
    const int nv = (E + 31) / 32;
    if (nv <= 1) return launch_topk_nv<1>(logits, part, split, bias, T, E, K, idx, gate, tie, counts, st);
    if (nv <= 2) return launch_topk_nv<2>(logits, part, split, bias, T, E, K, idx, gate, tie, counts, st);
    if (nv <= 4) return launch_topk_nv<4>(logits, part, split, bias, T, E, K, idx, gate, tie, counts, st);
    if (nv <= 8) return launch_topk_nv<8>(logits, part, split, bias, T, E, K, idx, gate, tie, counts, st);
    if (nv <= 16) return launch_topk_nv<16>(logits, part, split, bias, T, E, K, idx, gate, tie, counts, st);
    return launch_topk_nv<32>(logits, part, split, bias, T, E, K, idx, gate, tie, counts, st);
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Allocation-free router entry point.
//
// Some callers cannot call cudaMalloc at the moment they route tokens: a
// serving engine that hands all device memory to its own pool up front, a
// runtime whose allocator is not reachable from the thread that launches
// the layer, or code that must not allocate between two points it has
// measured or captured.  moe_route_noalloc serves them: it takes no
// workspace and keeps the [T, E] logits in a fixed array that lives in the
// library's own device memory (every GPU that loads the library holds these
// 4 MB until the process exits).
//
// In host code the array's name is only a host-side stand-in, so its device
// address is looked up with cudaGetSymbolAddress, once per device, with that
// device current, on the first call made there.  Every call shares the
// array and it keeps the last call's contents; two calls that overlap on the
// GPU (different streams, or different host threads on one device) race on
// it.  The array's first T * E floats hold the logits and the rest holds the
// split-K partial sums, as many splits as fit, which the selection kernel
// adds in a fixed order: repeated calls on the same input give identical
// results (no atomics; nothing read before it is written in the same call).
namespace moe {
namespace {

constexpr size_t kNoAllocMaxLogits = size_t(1) << 20;     // T * E limit (4 MB of float32)
static __device__ __align__(256) float g_noalloc_logits[kNoAllocMaxLogits];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_logits on the current device (set-up on first use).
int noalloc_scratch(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED_SHAPE;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_logits);
        if (e != cudaSuccess) return cuda_fail(e);
        g_noalloc_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_route_noalloc(const uint16_t* u, const float* centroids, const float* bias,
                                 int T, int d, int E, int K, int32_t* topk_idx, float* topk_gate,
                                 uint8_t* tie_flag, int32_t* counts, void* stream) {
    using namespace moe;
    if (T < 0 || d <= 0 || E <= 0 || K <= 0 || K > E || K > kMaxTopK || E > kMaxExperts)
        return MOE_ERR_INVALID_ARG;
    if (d % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!counts || !centroids || !bias) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!u || !topk_idx || !topk_gate || !tie_flag)) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(u) | reinterpret_cast<uintptr_t>(centroids)) & 15u)
        return MOE_ERR_MISALIGNED;
    if ((size_t)T * (size_t)E > kNoAllocMaxLogits) return MOE_ERR_WORKSPACE;
    float* logits = nullptr;
    const int rc = noalloc_scratch(&logits);
    if (rc) return rc;
    const size_t TE = (size_t)T * (size_t)E;
    return launch_route(u, centroids, bias, T, d, E, K, topk_idx, topk_gate, tie_flag, counts,
                        logits, static_cast<cudaStream_t>(stream), logits + TE,
                        kNoAllocMaxLogits - TE);
}
