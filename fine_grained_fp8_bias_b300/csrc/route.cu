// Router: affinity logits, sigmoid, bias-steered top-K, gate normalisation.
//
// Source: "รายงานเชิงเทคนิคของ DeepSeek-V3" (xyznot.com/th/paper/2412.19437),
// Method §2: s_{i,t} = Sigmoid(u_t^T e_i); g'_{i,t} = s_{i,t} when
// s_{i,t} + b_i is among the top K_r of {s_{j,t} + b_j}, else 0; g is g'
// normalised.  "Deepseek V3 国货之光 开源之光" (databean.com.cn), section
// "Auxiliary-Loss-Free Load Balancing": the bias b_i only steers which
// experts are chosen; the gate values use the unbiased s.
//
// Logits l = u E^T run on the tensor cores: every float32 centroid value c
// is split exactly into three bfloat16 pieces (hi = bf16(c), mid =
// bf16(c - hi), lo = c - hi - mid; 3 x 8 significand bits hold all 24 of
// float32), the bfloat16 token rows are used as they are, and a
// tcgen05.mma.kind::f16 GEMM sums the exact products in float32 TMEM over
// the whole of d; the epilogue adds the three pieces of each expert.  A
// float32 CUDA-core GEMM (logits_kernel) serves callers without the split
// workspace.  Then one warp per token does sigmoid, selection and gates.
// Selection order: descending s + b, equal scores broken by the lower expert
// index.  Near-tie flag: the K-th and (K+1)-th biased scores differ by less
// than 1e-6.
#include <cfloat>
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int LT = 64;   // tokens per logits tile
constexpr int LE = 64;   // experts per logits tile
constexpr int LK = 32;   // d per smem step

// l[t, e] (+)= sum_{j in this block's d-range} u[t, j] * c[e, j].
// 256 threads, each computing a 4 x 4 patch of the 64 x 64 tile.  With
// split > 1 (few tokens) every block adds its partial sum atomically into a
// zeroed l.
__global__ void __launch_bounds__(256) logits_kernel(const uint16_t* __restrict__ u,
                                                     const float* __restrict__ c, int T, int d,
                                                     int E, int split, float* __restrict__ l) {
    __shared__ __align__(16) float us[LK][LT + 4];
    __shared__ __align__(16) float cs[LK][LE + 4];
    const int tid = threadIdx.x;
    const int t0 = blockIdx.x * LT, e0 = blockIdx.y * LE;
    const int steps = d / LK;
    const int s_begin = (int)((long long)steps * blockIdx.z / split);
    const int s_end = (int)((long long)steps * (blockIdx.z + 1) / split);
    const int ty = tid >> 4, tx = tid & 15;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
    const int lrow = tid >> 2;          // 0..63: token (or expert) loaded by this thread
    const int lk = (tid & 3) * 8;       // 8 consecutive k
    for (int s = s_begin; s < s_end; ++s) {
        const int k0 = s * LK;
        {
            const int t = t0 + lrow;
            float v[8];
            if (t < T) {
                uint4 raw = *reinterpret_cast<const uint4*>(u + (size_t)t * d + k0 + lk);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[2 * i] = bf16_bits_to_float(static_cast<uint16_t>(w[i] & 0xFFFFu));
                    v[2 * i + 1] = bf16_bits_to_float(static_cast<uint16_t>(w[i] >> 16));
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) us[lk + i][lrow] = v[i];
        }
        {
            const int e = e0 + lrow;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (e < E) {
                const float4* p = reinterpret_cast<const float4*>(c + (size_t)e * d + k0 + lk);
                a = p[0];
                b = p[1];
            }
            cs[lk + 0][lrow] = a.x; cs[lk + 1][lrow] = a.y; cs[lk + 2][lrow] = a.z; cs[lk + 3][lrow] = a.w;
            cs[lk + 4][lrow] = b.x; cs[lk + 5][lrow] = b.y; cs[lk + 6][lrow] = b.z; cs[lk + 7][lrow] = b.w;
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < LK; ++k) {
            const float4 a = *reinterpret_cast<const float4*>(&us[k][ty * 4]);
            const float4 b = *reinterpret_cast<const float4*>(&cs[k][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
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
            if (split > 1)
                atomicAdd(&l[(size_t)t * E + e], acc[i][j]);
            else
                l[(size_t)t * E + e] = acc[i][j];
        }
    }
}


// ------------------------------------------------------- tensor-core logits
constexpr int RT_M = 128;                 // tokens per tile
constexpr int RT_EXP = 64;                // experts per tile
constexpr int RT_N = 3 * RT_EXP;          // MMA N: three pieces per expert
constexpr int RT_K = 64;                  // bf16 elements per 128-byte smem row
constexpr int RT_STAGES = 4;
constexpr int RT_SMEM_A = RT_M * 128;
constexpr int RT_SMEM_B = RT_N * 128;
constexpr int RT_STAGE = RT_SMEM_A + RT_SMEM_B;
constexpr int RT_THREADS = 192;           // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr uint32_t RT_TMEM_COLS = 256;

struct alignas(8) RtCtl {
    uint64_t full[RT_STAGES];
    uint64_t empty[RT_STAGES];
    uint64_t done;
    uint32_t tmem_base;
    int abort;
};
constexpr size_t RT_SMEM_BYTES = 1024 + (size_t)RT_STAGES * RT_STAGE + sizeof(RtCtl);

// c = hi + mid + lo exactly (float32 subtractions of a value and its
// bfloat16 rounding are exact).  out row 3e + j holds piece j of expert e.
__global__ void split_centroids_kernel(const float* __restrict__ c, int E, int d,
                                       __nv_bfloat16* __restrict__ out) {
    const size_t n = (size_t)E * d;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const float v = c[i];
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const float r1 = v - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);
        const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
        const size_t e = i / d, j = i % d;
        out[(3 * e + 0) * d + j] = hi;
        out[(3 * e + 1) * d + j] = mid;
        out[(3 * e + 2) * d + j] = lo;
    }
}

// One tile of 128 tokens x 64 experts over the k-steps [kb0, kb1) of d.
// split > 1: partial sums are added atomically into a zeroed l.
__global__ void __launch_bounds__(RT_THREADS, 1)
    logits_tc_kernel(const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmC,
                     int T, int d, int E, int split, float* __restrict__ l, int32_t* status) {
    using namespace tc;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    RtCtl* ctl = reinterpret_cast<RtCtl*>(smem + (size_t)RT_STAGES * RT_STAGE);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * RT_M, e0 = blockIdx.y * RT_EXP;
    const int steps = d / RT_K;
    const int kb0 = (int)((long long)steps * blockIdx.z / split);
    const int kb1 = (int)((long long)steps * (blockIdx.z + 1) / split);

    if (warp == 0 && lane == 0) {
        ctl->abort = 0;
        for (int s = 0; s < RT_STAGES; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        mbar_init(&ctl->done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tmU);
        tma_prefetch_desc(&tmC);
    } else if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&ctl->tmem_base)),
                     "r"(RT_TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            uint32_t it = 0;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = it % RT_STAGES;
                if (!mbar_wait(&ctl->empty[s], ((it / RT_STAGES) & 1) ^ 1, &ctl->abort, status)) break;
                uint8_t* sA = smem + (size_t)s * RT_STAGE;
                mbar_expect_tx(&ctl->full[s], RT_STAGE);
                tma_load_2d(sA, &tmU, &ctl->full[s], kb * RT_K, t0);
                tma_load_2d(sA + RT_SMEM_A, &tmC, &ctl->full[s], kb * RT_K, 3 * e0);
            }
            const uint32_t first = it > (uint32_t)RT_STAGES ? it - RT_STAGES : 0;
            for (uint32_t j = first; j < it; ++j) mbar_drain(&ctl->full[j % RT_STAGES], (j / RT_STAGES) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(RT_M, RT_N);
            uint32_t it = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = it % RT_STAGES;
                if (!mbar_wait(&ctl->full[s], (it / RT_STAGES) & 1, &ctl->abort, status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t a0 = smem_u32(smem + (size_t)s * RT_STAGE);
                const uint32_t b0 = a0 + RT_SMEM_A;
#pragma unroll
                for (int k = 0; k < RT_K / 16; ++k)
                    mma_bf16(tmem_base, sdesc_sw128(a0 + k * 32), sdesc_sw128(b0 + k * 32), idesc,
                             (kb > kb0 || k > 0) ? 1u : 0u);
                mma_commit(&ctl->empty[s]);
            }
            // committed in every case, so teardown can wait for the MMAs in flight
            mma_commit(&ctl->done);
            if (!ok) atomicExch(&ctl->abort, 1);
        }
    } else {
        // epilogue: thread (warp, lane) owns token row 32 * (warp % 4) + lane
        const int quarter = warp & 3;
        const int t = t0 + quarter * 32 + lane;
        if (warp_wait(&ctl->done, 0, &ctl->abort, status)) {
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll
            for (int c = 0; c < RT_N / 96; ++c) {
                // 96 columns = 32 experts x 3 pieces
                uint32_t a[32], b[32], g[32];
                tmem_ld32_nowait(tbase + c * 96, a);
                tmem_ld32_nowait(tbase + c * 96 + 32, b);
                tmem_ld32_nowait(tbase + c * 96 + 64, g);
                tmem_ld_wait(a);
                reg_after_wait(b);
                reg_after_wait(g);
                float v[96];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    v[i] = __uint_as_float(a[i]);
                    v[32 + i] = __uint_as_float(b[i]);
                    v[64 + i] = __uint_as_float(g[i]);
                }
                if (t < T) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int e = e0 + c * 32 + j;
                        if (e < E) {
                            const float x = (v[3 * j] + v[3 * j + 1]) + v[3 * j + 2];
                            if (split > 1)
                                atomicAdd(&l[(size_t)t * E + e], x);
                            else
                                l[(size_t)t * E + e] = x;
                        }
                    }
                }
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 1) {
        // every MMA has completed (done, or the drained empty barriers) and every
        // TMEM read is finished before the release
        if (lane == 0) mbar_drain(&ctl->done, 0);
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(RT_TMEM_COLS));
    }
}

// Larger score first; equal scores: lower expert index first.
__device__ __forceinline__ bool better(float za, int ia, float zb, int ib) {
    return za > zb || (za == zb && ia < ib);
}

// One warp per token.  Lane L holds experts L, L + 32, ... (NV per lane).
template <int NV>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ l,
                                                   const float* __restrict__ bias, int T, int E,
                                                   int K, int32_t* __restrict__ idx,
                                                   float* __restrict__ gate,
                                                   uint8_t* __restrict__ tie,
                                                   int32_t* __restrict__ counts) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    float s[NV], z[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const int e = j * 32 + lane;
        if (e < E) {
            const float x = l[(size_t)t * E + e];
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
void launch_topk_nv(const float* l, const float* bias, int T, int E, int K, int32_t* idx,
                    float* gate, uint8_t* tie, int32_t* counts, cudaStream_t st) {
    const int warps = 8;
    topk_kernel<NV><<<(T + warps - 1) / warps, warps * 32, 0, st>>>(l, bias, T, E, K, idx, gate,
                                                                     tie, counts);
}

}  // namespace

int launch_route(const uint16_t* u, const float* cent, const float* bias, int T, int d, int E,
                 int K, int32_t* idx, float* gate, uint8_t* tie, int32_t* counts, float* logits,
                 cudaStream_t st, uint16_t* cent_split, int32_t* status) {
    cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)E, st);
    if (e != cudaSuccess) return cuda_fail(e);
    if (T == 0) return MOE_OK;
    int rc;
    if (cent_split) {
        // tensor-core logits
        static std::once_flag once;
        std::call_once(once, [] {
            cudaFuncSetAttribute(logits_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)RT_SMEM_BYTES);
        });
        __nv_bfloat16* cs = reinterpret_cast<__nv_bfloat16*>(cent_split);
        split_centroids_kernel<<<148 * 4, 256, 0, st>>>(cent, E, d, cs);
        if ((rc = check_launch())) return rc;
        CUtensorMap mU, mC;
        if ((rc = tc::make_map_2d(&mU, u, (uint64_t)T, (uint64_t)d, 2, RT_M, RT_K))) return rc;
        if ((rc = tc::make_map_2d(&mC, cs, (uint64_t)3 * E, (uint64_t)d, 2, RT_N, RT_K))) return rc;
        const int gx = (T + RT_M - 1) / RT_M, gy = (E + RT_EXP - 1) / RT_EXP;
        const int steps = d / RT_K;
        int split = 1;
        while (gx * gy * split * 2 <= 2 * 148 && split * 2 <= steps / 4 && gx * gy * split < 74)
            split *= 2;
        if (split > 1) {
            e = cudaMemsetAsync(logits, 0, sizeof(float) * (size_t)T * E, st);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        logits_tc_kernel<<<dim3(gx, gy, split), RT_THREADS, RT_SMEM_BYTES, st>>>(
            mU, mC, T, d, E, split, logits, status);
        if ((rc = check_launch())) return rc;
    } else {
        const int gx = (T + LT - 1) / LT, gy = (E + LE - 1) / LE;
        int split = 1;
        const int target = 2 * 148;
        while (gx * gy * split < target && split * 2 <= d / LK / 4) split *= 2;
        if (split > 1) {
            e = cudaMemsetAsync(logits, 0, sizeof(float) * (size_t)T * E, st);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        logits_kernel<<<dim3(gx, gy, split), 256, 0, st>>>(u, cent, T, d, E, split, logits);
        if ((rc = check_launch())) return rc;
    }
    const int nv = (E + 31) / 32;
    if (nv <= 1) launch_topk_nv<1>(logits, bias, T, E, K, idx, gate, tie, counts, st);
    else if (nv <= 2) launch_topk_nv<2>(logits, bias, T, E, K, idx, gate, tie, counts, st);
    else if (nv <= 4) launch_topk_nv<4>(logits, bias, T, E, K, idx, gate, tie, counts, st);
    else if (nv <= 8) launch_topk_nv<8>(logits, bias, T, E, K, idx, gate, tie, counts, st);
    else if (nv <= 16) launch_topk_nv<16>(logits, bias, T, E, K, idx, gate, tie, counts, st);
    else launch_topk_nv<32>(logits, bias, T, E, K, idx, gate, tie, counts, st);
    return check_launch();
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
// array and it keeps the last call's contents: the split-K path clears the
// logits before it accumulates into them, and two calls that overlap on the
// GPU (different streams, or different host threads on one device) race on
// it.
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
    return launch_route(u, centroids, bias, T, d, E, K, topk_idx, topk_gate, tie_flag, counts,
                        logits, static_cast<cudaStream_t>(stream));
}
