// Router of moe_route: affinity, sigmoid, bias-steered top-K and gates, with
// the logits screened on the tensor cores and recomputed exactly only where
// the selection depends on them.
//
// Source: "รายงานเชิงเทคนิคของ DeepSeek-V3" (xyznot.com/th/paper/2412.19437),
// Method §2: s_{i,t} = Sigmoid(u_t^T e_i); expert i is selected for token t
// when s_{i,t} + b_i is among the K_r largest of {s_{j,t} + b_j}; the gates
// are the selected s normalised to sum 1.  "Deepseek V3 国货之光 开源之光"
// (databean.com.cn), "Auxiliary-Loss-Free Load Balancing": b only steers the
// choice, the gates use the unbiased s.
//
// The selection has a near-tie band 1e-6 wide, so the scores it compares must
// be close to exact; only about K of the E logits of a token matter, though.
//   1. split_centroids: c = hi + mid + r with hi = bf16(c), mid = bf16(c - hi)
//      (|r| <= 2^-16 |c| elementwise), and the largest centroid norm.
//   2. logits_tc: l~ = u hi^T + u mid^T on the tensor cores
//      (tcgen05.mma.kind::f16, bf16 operands, float32 accumulation in TMEM),
//      split over d when there are few token tiles; partial sums to [split][T][E].
//   3. screen (one warp per token): |l~_e - l_e| is bounded by
//      gamma |u_t| |c_e| (gamma = 2^-11 covers the split remainder and an error
//      of one float32 ulp of the running sum per MMA instruction, with twofold
//      headroom), and sigmoid has slope at most 1/4, so every biased score z_e
//      lies in [lo_e, hi_e] around its estimate.  The K-th largest z is at
//      least L_K, the K-th largest lo; an expert with hi_e < L_K - 2e-6 can
//      neither be selected nor lie within 2e-6 of the K-th score, and every
//      other expert is a candidate.
//   4. exact: the candidates' logits recomputed on CUDA cores with
//      compensated summation (32-term FMA chains added with TwoSum), grouped
//      by expert so that each centroid row is read once per block.
//   5. select (one warp per token): selection, gates and tie flag from the
//      exact logits.  A token with more than 64 candidates (degenerate inputs:
//      many equal scores) recomputes all E there.
// Selection order: descending s + b, equal scores broken by the lower expert
// index.  Near-tie flag: the K-th and (K+1)-th biased scores differ by less
// than 1e-6.
#include <cfloat>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {
using namespace tc;

constexpr int RT_M = 128;                           // tokens per tile
constexpr int RT_N = 128;                           // experts per tile
constexpr int RT_K = 64;                            // bf16 elements per slab (128 bytes)
constexpr int RT_STAGES = 4;
constexpr int RT_SMEM_A = RT_M * RT_K * 2;          // 16 KB
constexpr int RT_SMEM_B = RT_N * RT_K * 2;          // 16 KB per centroid piece
constexpr int RT_STAGE = RT_SMEM_A + 2 * RT_SMEM_B; // 48 KB
constexpr int RT_THREADS = 128;
constexpr uint32_t RT_TMEM_COLS = 128;
constexpr int CAND_CAP = 64;
constexpr float GAMMA = 0x1p-11f;
constexpr int SEL_WARPS = 4;                        // warps per token in select_refine

struct RtCtl {
    uint64_t full[RT_STAGES];
    uint64_t empty[RT_STAGES];
    uint64_t done;
    uint32_t tmem_base;
    int abort;
};
constexpr size_t RT_SMEM_BYTES = 1024 + (size_t)RT_STAGES * RT_STAGE + sizeof(RtCtl);

// Workspace: header (status word), centroid norms, hi, mid, partial logits.
struct RouteWs {
    size_t status, norms, hi, mid, part, cand_n, cand_e, exact, bucket_cnt, bucket, total;
    int split;
};

int route_split(int T, int E, int d) {
    const int tiles = ((T + RT_M - 1) / RT_M) * ((E + RT_N - 1) / RT_N);
    const int slabs = d / RT_K;
    int split = 1;
    while (tiles * split * 2 <= 148 && split * 2 <= slabs / 8) split *= 2;
    return split;
}

RouteWs route_ws(int T, int d, int E) {
    RouteWs w{};
    w.split = route_split(T, E, d);
    w.status = 0;
    w.norms = 256;
    w.hi = align_up(w.norms + sizeof(float) * (size_t)E, 256);
    w.mid = align_up(w.hi + (size_t)E * d * 2, 256);
    w.part = align_up(w.mid + (size_t)E * d * 2, 256);
    w.cand_n = align_up(w.part + sizeof(float) * (size_t)w.split * T * E, 256);
    w.cand_e = align_up(w.cand_n + sizeof(int32_t) * (size_t)T, 256);
    w.exact = align_up(w.cand_e + sizeof(int32_t) * (size_t)T * CAND_CAP, 256);
    w.bucket_cnt = align_up(w.exact + sizeof(float) * (size_t)T * CAND_CAP, 256);
    w.bucket = align_up(w.bucket_cnt + sizeof(int32_t) * (size_t)E, 256);
    w.total = align_up(w.bucket + sizeof(int32_t) * (size_t)E * T, 256);
    return w;
}

// Error-free sum (Knuth's TwoSum): s + err == a + b exactly.
__device__ __forceinline__ float two_sum(float a, float b, float& err) {
    const float s = a + b;
    const float bb = s - a;
    err = (a - (s - bb)) + (b - bb);
    return s;
}

__device__ __forceinline__ float sigmoid(float x) { return __fdiv_rn(1.0f, 1.0f + expf(-x)); }

// Larger score first; equal scores: lower expert index first.
__device__ __forceinline__ bool better(float za, int ia, float zb, int ib) {
    return za > zb || (za == zb && ia < ib);
}

// ------------------------------------------------------------ 1. split
// One block per expert row: hi/mid pieces and |c_e| (times 1 + 2^-20 for its
// own rounding) to norms[e].
constexpr int SPLIT_THREADS = 256;
// Block e also zeroes zero0[e] and zero1[e] (nullable): the counts and the
// expert bucket sizes that later kernels of the same call add into.
__global__ void __launch_bounds__(SPLIT_THREADS) split_centroids_kernel(
    const float* __restrict__ c, int E, int d, uint16_t* __restrict__ hi,
    uint16_t* __restrict__ mid, float* __restrict__ norms, int32_t* __restrict__ zero0,
    int32_t* __restrict__ zero1) {
    __shared__ float wsum[SPLIT_THREADS / 32];
    griddep_wait();
    griddep_launch();
    const int e = blockIdx.x;
    if (threadIdx.x == 0) {
        if (zero0) zero0[e] = 0;
        if (zero1) zero1[e] = 0;
    }
    float ss = 0.0f;
    for (int j = threadIdx.x * 4; j < d; j += SPLIT_THREADS * 4) {
        const size_t at = (size_t)e * d + j;
        const float4 v = *reinterpret_cast<const float4*>(c + at);
        const float x[4] = {v.x, v.y, v.z, v.w};
        uint16_t h[4], m[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat16 bh = __float2bfloat16_rn(x[i]);
            const __nv_bfloat16 bm = __float2bfloat16_rn(x[i] - __bfloat162float(bh));
            h[i] = __bfloat16_as_ushort(bh);
            m[i] = __bfloat16_as_ushort(bm);
            ss = fmaf(x[i], x[i], ss);
        }
        *reinterpret_cast<uint2*>(hi + at) =
            make_uint2(h[0] | ((uint32_t)h[1] << 16), h[2] | ((uint32_t)h[3] << 16));
        *reinterpret_cast<uint2*>(mid + at) =
            make_uint2(m[0] | ((uint32_t)m[1] << 16), m[2] | ((uint32_t)m[3] << 16));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.0f;
        for (int w = 0; w < SPLIT_THREADS / 32; ++w) t += wsum[w];
        norms[e] = sqrtf(t) * (1.0f + 0x1p-20f);
    }
}

// ------------------------------------------------------------ 2. logits_tc
// One CTA: 128 tokens x 128 experts over the slabs [kb0, kb1) of d.  Warp 0
// lane 0 loads (TMA, 128-byte swizzle), warp 1 lane 0 issues the MMAs (both
// pieces into one TMEM accumulator), then all four warps read TMEM (thread
// (warp, lane) owns token row 32 warp + lane) and store the partial sums.
__global__ void __launch_bounds__(RT_THREADS, 1)
    logits_tc_kernel(const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmH,
                     const __grid_constant__ CUtensorMap tmM, int T, int d, int E, int split,
                     float* __restrict__ part, int32_t* status) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    griddep_wait();
    griddep_launch();
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    RtCtl* ctl = reinterpret_cast<RtCtl*>(smem + (size_t)RT_STAGES * RT_STAGE);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * RT_M, e0 = blockIdx.y * RT_N;
    const int slabs = d / RT_K;
    const int kb0 = (int)((long long)slabs * blockIdx.z / split);
    const int kb1 = (int)((long long)slabs * (blockIdx.z + 1) / split);

    if (warp == 0 && lane == 0) {
        ctl->abort = 0;
        for (int s = 0; s < RT_STAGES; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        mbar_init(&ctl->done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tmU);
        tma_prefetch_desc(&tmH);
        tma_prefetch_desc(&tmM);
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
                tma_load_2d(sA + RT_SMEM_A, &tmH, &ctl->full[s], kb * RT_K, e0);
                tma_load_2d(sA + RT_SMEM_A + RT_SMEM_B, &tmM, &ctl->full[s], kb * RT_K, e0);
            }
            // no copy may still be landing when the CTA exits
            const uint32_t first = it > (uint32_t)RT_STAGES ? it - RT_STAGES : 0;
            for (uint32_t j = first; j < it; ++j) mbar_drain(&ctl->full[j % RT_STAGES], (j / RT_STAGES) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(RT_M, RT_N);
            uint32_t it = 0;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = it % RT_STAGES;
                if (!mbar_wait(&ctl->full[s], (it / RT_STAGES) & 1, &ctl->abort, status)) break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(smem + (size_t)s * RT_STAGE);
                const uint32_t bh = a0 + RT_SMEM_A, bm = bh + RT_SMEM_B;
#pragma unroll
                for (int k = 0; k < RT_K / 16; ++k)
                    mma_bf16(tmem_base, sdesc_sw128(a0 + k * 32), sdesc_sw128(bh + k * 32), idesc,
                             (kb > kb0 || k > 0) ? 1u : 0u);
#pragma unroll
                for (int k = 0; k < RT_K / 16; ++k)
                    mma_bf16(tmem_base, sdesc_sw128(a0 + k * 32), sdesc_sw128(bm + k * 32), idesc, 1u);
                mma_commit(&ctl->empty[s]);
            }
            // committed in every case, so the epilogue and the teardown can wait
            // for the MMAs in flight
            mma_commit(&ctl->done);
        }
    }
    __syncwarp();
    // epilogue: every warp, after the accumulator is complete
    if (warp_wait(&ctl->done, 0, &ctl->abort, status)) {
        tc_fence_after();
        const int t = t0 + warp * 32 + lane;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16);
        float* dst = part + ((size_t)blockIdx.z * T + (t < T ? t : 0)) * E;
#pragma unroll
        for (int c = 0; c < RT_N / 32; ++c) {
            uint32_t v[32];
            tmem_ld32_nowait(taddr + c * 32, v);
            tmem_ld_wait(v);
            if (t < T) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int e = e0 + c * 32 + i;
                    if (e < E) dst[e] = __uint_as_float(v[i]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0) mbar_drain(&ctl->done, 0);
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(RT_TMEM_COLS));
    }
}

// ------------------------------------------------------------ 3. select_refine
// l = u_t . c_e with compensated summation.  Lane L takes elements
// 128 i + 4 L .. + 3; each 32-product FMA chain starts from zero and is added
// into (acc, cmp) with TwoSum; the lanes' pairs are then combined with TwoSum
// too (the xor butterfly leaves the same value in every lane).  The centroid
// loads of the next 8 blocks are issued before the current ones are used.
__device__ __forceinline__ float exact_dot(const uint16_t* ut, const float* __restrict__ crow,
                                           int d, int lane) {
    const int nblk = d / 128;
    float acc = 0.0f, cmp = 0.0f;
    float4 nxt[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
        if (q < nblk) nxt[q] = __ldg(reinterpret_cast<const float4*>(crow + q * 128 + lane * 4));
    for (int i = 0; i < nblk; i += 8) {
        float4 cv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) cv[q] = nxt[q];
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (i + 8 + q < nblk)
                nxt[q] = __ldg(reinterpret_cast<const float4*>(crow + (i + 8 + q) * 128 + lane * 4));
        float p = 0.0f;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (i + q < nblk) {
                const uint2 uv = *reinterpret_cast<const uint2*>(ut + (i + q) * 128 + lane * 4);
                p = fmaf(bf16_bits_to_float(static_cast<uint16_t>(uv.x & 0xFFFFu)), cv[q].x, p);
                p = fmaf(bf16_bits_to_float(static_cast<uint16_t>(uv.x >> 16)), cv[q].y, p);
                p = fmaf(bf16_bits_to_float(static_cast<uint16_t>(uv.y & 0xFFFFu)), cv[q].z, p);
                p = fmaf(bf16_bits_to_float(static_cast<uint16_t>(uv.y >> 16)), cv[q].w, p);
            }
        }
        float err;
        acc = two_sum(acc, p, err);
        cmp += err;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float oa = __shfl_xor_sync(0xffffffffu, acc, off);
        const float oc = __shfl_xor_sync(0xffffffffu, cmp, off);
        float err;
        acc = two_sum(acc, oa, err);
        cmp = (cmp + oc) + err;
    }
    return acc + cmp;
}

// The K-th largest value of z over the warp (lane L holds experts L + 32 j).
template <int NV>
__device__ __forceinline__ float kth_largest(const float (&z)[NV], int E, int K, int lane) {
    unsigned taken = 0;
    float zk = -FLT_MAX;
    for (int k = 0; k < K; ++k) {
        float bz = -FLT_MAX;
        int be = 0x7fffffff, bj = -1;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int e = j * 32 + lane;
            if (e < E && !(taken >> j & 1u) && better(z[j], e, bz, be)) { bz = z[j]; be = e; bj = j; }
        }
        float wz = bz;
        int we = be;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float oz = __shfl_xor_sync(0xffffffffu, wz, off);
            const int oe = __shfl_xor_sync(0xffffffffu, we, off);
            if (better(oz, oe, wz, we)) { wz = oz; we = oe; }
        }
        if (we == be && bj >= 0) taken |= 1u << bj;
        zk = wz;
    }
    return zk;
}

// ------------------------------------------------------------ 3. screen / exact / select
// The exact recomputation reorganised by expert, so that a centroid row read
// once serves every token that has the expert as a candidate:
//   screen  one warp per token: bounds of every biased score around its
//           estimate, the candidates (in expert order) to cand_e[t][k], and
//           each (token, slot) appended to its expert's bucket;
//   exact   the buckets cut into equal runs of pairs; a block loads each
//           expert's centroid row into shared memory once and its warps
//           compute the candidates' logits (same compensated summation as
//           exact_dot) into exact[t][k];
//   select  one warp per token: sigmoid, selection, gates, tie flag, counts.
// The order of the entries inside a bucket depends on timing, but every
// (token, expert) logit is computed the same way wherever it lands, so the
// results do not.  A token with more than CAND_CAP candidates (degenerate
// inputs) computes all E logits in the select kernel.

// |u_t|^2 by one warp (lane L takes 8 consecutive elements of every 256);
// eight rows' worth of loads are issued before any is used.
__device__ __forceinline__ float warp_sumsq_bf16(const uint16_t* ut, int d, int lane) {
    float ss = 0.0f;
    for (int j0 = lane * 8; j0 < d; j0 += 8 * 256) {
        uint4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (j0 + q * 256 < d) v[q] = __ldg(reinterpret_cast<const uint4*>(ut + j0 + q * 256));
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (j0 + q * 256 >= d) break;
            const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float lo = bf16_bits_to_float(static_cast<uint16_t>(w[i] & 0xFFFFu));
                const float hi = bf16_bits_to_float(static_cast<uint16_t>(w[i] >> 16));
                ss = fmaf(lo, lo, fmaf(hi, hi, ss));
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    return ss;
}

constexpr int SCR_WARPS = 8;
template <int NV>
__global__ void __launch_bounds__(SCR_WARPS * 32) screen_kernel(
    const uint16_t* __restrict__ u, const float* __restrict__ bias, const float* __restrict__ part,
    int split, int T, int d, int E, int K, const float* __restrict__ norms,
    int32_t* __restrict__ cand_n, int32_t* __restrict__ cand_e, int32_t* __restrict__ bucket_cnt,
    int32_t* __restrict__ bucket) {
    griddep_wait();
    griddep_launch();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * SCR_WARPS + (threadIdx.x >> 5);
    if (t >= T) return;
    const float ss = warp_sumsq_bf16(u + (size_t)t * d, d, lane);
    const float gu = GAMMA * sqrtf(ss);
    float lo[NV], hi[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const int e = j * 32 + lane;
        if (e < E) {
            float l = 0.0f;
            for (int q = 0; q < split; ++q) l += part[((size_t)q * T + t) * E + e];
            const float za = sigmoid(l) + bias[e];
            const float eps = 0.25f * gu * norms[e] + 1e-6f + 0x1p-22f * (fabsf(za) + 1.0f);
            lo[j] = za - eps;
            hi[j] = za + eps;
        } else {
            lo[j] = hi[j] = -FLT_MAX;
        }
    }
    const float LK = kth_largest(lo, E, K, lane);
    unsigned cand = 0;
#pragma unroll
    for (int j = 0; j < NV; ++j)
        if (j * 32 + lane < E && hi[j] >= LK - 2e-6f) cand |= 1u << j;
    int n = __popc(cand);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) n += __shfl_xor_sync(0xffffffffu, n, off);
    if (n > CAND_CAP) {                         // degenerate: the select kernel takes all E
        if (lane == 0) cand_n[t] = -1;
        return;
    }
    int base = 0;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const unsigned m = __ballot_sync(0xffffffffu, (cand >> j) & 1u);
        if ((cand >> j) & 1u) {
            const int e = j * 32 + lane;
            const int k = base + __popc(m & ((1u << lane) - 1u));
            cand_e[(size_t)t * CAND_CAP + k] = e;
            const int pos = atomicAdd(&bucket_cnt[e], 1);
            bucket[(size_t)e * T + pos] = t * CAND_CAP + k;
        }
        base += __popc(m);
    }
    if (lane == 0) cand_n[t] = n;
}

// l = u_t . c_e as exact_dot, with the token row read from global memory and
// the centroid row from shared memory.
__device__ __forceinline__ float exact_dot_gs(const uint16_t* __restrict__ ut, const float* cs,
                                              int d, int lane) {
    const int nblk = d / 128;
    float acc = 0.0f, cmp = 0.0f;
    for (int i = 0; i < nblk; i += 16) {
        uint2 uv[16];                           // sixteen blocks' loads in flight
#pragma unroll
        for (int q = 0; q < 16; ++q)
            if (i + q < nblk) uv[q] = __ldg(reinterpret_cast<const uint2*>(ut + (i + q) * 128 + lane * 4));
#pragma unroll
        for (int h = 0; h < 2; ++h) {           // two chains of eight blocks, in order
            if (i + 8 * h >= nblk) break;
            float p = 0.0f;
#pragma unroll
            for (int q = 8 * h; q < 8 * h + 8; ++q) {
                if (i + q < nblk) {
                    const float4 cv = *reinterpret_cast<const float4*>(cs + (i + q) * 128 + lane * 4);
                    p = fmaf(bf16_bits_to_float(static_cast<uint16_t>(uv[q].x & 0xFFFFu)), cv.x, p);
                    p = fmaf(bf16_bits_to_float(static_cast<uint16_t>(uv[q].x >> 16)), cv.y, p);
                    p = fmaf(bf16_bits_to_float(static_cast<uint16_t>(uv[q].y & 0xFFFFu)), cv.z, p);
                    p = fmaf(bf16_bits_to_float(static_cast<uint16_t>(uv[q].y >> 16)), cv.w, p);
                }
            }
            float err;
            acc = two_sum(acc, p, err);
            cmp += err;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float oa = __shfl_xor_sync(0xffffffffu, acc, off);
        const float oc = __shfl_xor_sync(0xffffffffu, cmp, off);
        float err;
        acc = two_sum(acc, oa, err);
        cmp = (cmp + oc) + err;
    }
    return acc + cmp;
}

constexpr int EX_WARPS = 8;
// Dynamic shared memory: the centroid row [d] float, then the bucket offsets [E + 1].
__global__ void __launch_bounds__(EX_WARPS * 32) exact_pairs_kernel(
    const uint16_t* __restrict__ u, const float* __restrict__ c, int T, int d, int E,
    const int32_t* __restrict__ bucket_cnt, const int32_t* __restrict__ bucket,
    float* __restrict__ exact) {
    extern __shared__ __align__(16) float ex_sm[];
    griddep_wait();
    griddep_launch();
    float* cs = ex_sm;
    int* offs = reinterpret_cast<int*>(ex_sm + d);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // exclusive scan of the bucket sizes (warp 0; E <= 1024)
    if (warp == 0) {
        int carry = 0;
        for (int b0 = 0; b0 < E; b0 += 32) {
            const int e = b0 + lane;
            const int v = e < E ? bucket_cnt[e] : 0;
            int incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            if (e < E) offs[e] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) offs[E] = carry;
    }
    __syncthreads();
    const int total = offs[E];
    const int per = (total + gridDim.x - 1) / gridDim.x;
    const int beg = min(total, (int)blockIdx.x * per);
    const int end = min(total, beg + per);
    if (beg >= end) return;
    // first expert whose bucket holds pair index beg
    int lo = 0, hi = E;                         // offs[lo] <= beg < offs[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (offs[mid] <= beg) lo = mid; else hi = mid;
    }
    for (int e = lo, i0 = beg; i0 < end; ++e) {
        const int s0 = max(i0, offs[e]), s1 = min(end, offs[e + 1]);
        if (s0 >= s1) continue;
        __syncthreads();                        // the previous row is no longer read
        for (int j = threadIdx.x * 4; j < d; j += EX_WARPS * 32 * 4)
            *reinterpret_cast<float4*>(cs + j) = __ldg(reinterpret_cast<const float4*>(c + (size_t)e * d + j));
        __syncthreads();
        for (int i = s0 + warp; i < s1; i += EX_WARPS) {
            const int code = bucket[(size_t)e * T + (i - offs[e])];
            const int t = code / CAND_CAP;
            const float l = exact_dot_gs(u + (size_t)t * d, cs, d, lane);
            if (lane == 0) exact[code] = l;
        }
        i0 = s1;
    }
}

constexpr int SEL2_WARPS = 8;
template <int NV>
__global__ void __launch_bounds__(SEL2_WARPS * 32) select_exact_kernel(
    const uint16_t* __restrict__ u, const float* __restrict__ c, const float* __restrict__ bias,
    int T, int d, int E, int K, const int32_t* __restrict__ cand_n,
    const int32_t* __restrict__ cand_e, const float* __restrict__ exact,
    int32_t* __restrict__ idx, float* __restrict__ gate, uint8_t* __restrict__ tie,
    int32_t* __restrict__ counts) {
    constexpr int NC = NV < 2 ? NV : 2;          // CAND_CAP = 64 candidates: two per lane
    griddep_wait();
    griddep_launch();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * SEL2_WARPS + (threadIdx.x >> 5);
    if (t >= T) return;
    const int n = cand_n[t];
    float s[NV], z[NV];
    int ex[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        s[j] = 0.0f;
        z[j] = -FLT_MAX;
        ex[j] = 0x7fffffff;
    }
    int nc;
    if (n >= 0) {                               // the candidates' exact logits
        nc = n;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
            const int k = j * 32 + lane;
            if (k < n) {
                const int e = cand_e[(size_t)t * CAND_CAP + k];
                const float sv = sigmoid(exact[(size_t)t * CAND_CAP + k]);
                s[j] = sv;
                z[j] = sv + bias[e];
                ex[j] = e;
            }
        }
    } else {                                    // every expert, exactly (degenerate inputs)
        nc = E;
        const uint16_t* ut = u + (size_t)t * d;
        for (int e = 0; e < E; ++e) {
            const float l = exact_dot(ut, c + (size_t)e * d, d, lane);
            const float sv = sigmoid(l);
#pragma unroll
            for (int j = 0; j < NV; ++j)
                if (e == j * 32 + lane) { s[j] = sv; z[j] = sv + bias[e]; ex[j] = e; }
        }
    }
    unsigned taken = 0;
    float my_s = 0.0f, ssum = 0.0f, zk = 0.0f, zk1 = -FLT_MAX;
    int my_e = -1;
    const int rounds = K < E ? K + 1 : K;
    for (int k = 0; k < rounds; ++k) {
        float bz = -FLT_MAX;
        int be = 0x7fffffff, bj = -1;
        float bs = 0.0f;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            if (j * 32 + lane < nc && !(taken >> j & 1u) && better(z[j], ex[j], bz, be)) {
                bz = z[j]; be = ex[j]; bj = j; bs = s[j];
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
        if (we == be && bj >= 0) taken |= 1u << bj;
        if (k < K) {
            ssum += ws;                                  // same order in every lane
            if (lane == k) { my_e = we; my_s = ws; }
            if (k == K - 1) zk = wz;
        } else {
            zk1 = wz;                                    // -FLT_MAX: no candidate left
        }
    }
    if (lane < K) {
        idx[(size_t)t * K + lane] = my_e;
        gate[(size_t)t * K + lane] = __fdiv_rn(my_s, ssum);
        atomicAdd(&counts[my_e], 1);
    }
    if (lane == 0) tie[t] = (K < E && (zk - zk1) < 1e-6f) ? 1 : 0;
}

// ------------------------------------------------------------ 3b. grouped
// Group-limited selection: experts form n_groups contiguous groups of gs; a
// group's score is the float32 sum, largest first, of its group_topk best z;
// the topk_groups best groups are kept (equal: lower group index); top-K by z
// among their experts.  Flagged as a near tie also when the last kept and the
// next group score differ by less than 1e-6.
// Two exact rounds: (A) in every group whose estimated score could reach the
// cut, the experts that could be among its best group_topk; the kept groups
// follow from exact scores.  (B) in the kept groups, the experts within the
// band of the K-th estimated score.  Lane g of warp 0 scans group g.
// Shared memory: u_t [d] bf16, then zlo, zhi, zex, sex [32 NV] float (bounds
// of z around its estimate, exact z and s by expert; zex is NaN until
// computed), and the work list [32 NV] int.  A group's score lies between the
// sum of its group_topk largest lower bounds and that of its group_topk
// largest upper bounds.
template <int NV>
__global__ void __launch_bounds__(SEL_WARPS * 32) select_refine_grouped_kernel(
    const uint16_t* __restrict__ u, const float* __restrict__ c, const float* __restrict__ bias,
    const float* __restrict__ part, int split, int T, int d, int E, int K, int n_groups,
    int topk_groups, int group_topk, const float* __restrict__ norms,
    int32_t* __restrict__ idx, float* __restrict__ gate, uint8_t* __restrict__ tie,
    int32_t* __restrict__ counts) {
    griddep_wait();
    griddep_launch();
    extern __shared__ __align__(16) uint8_t sel_sm[];
    __shared__ float red[SEL_WARPS];
    __shared__ int n_work;
    __shared__ int all_mode;
    __shared__ int gtie_sh;
    uint16_t* ut = reinterpret_cast<uint16_t*>(sel_sm);
    float* zlo = reinterpret_cast<float*>(sel_sm + (size_t)d * 2);
    float* zhi = zlo + NV * 32;
    float* zex = zhi + NV * 32;
    float* sex = zex + NV * 32;
    int* work = reinterpret_cast<int*>(sex + NV * 32);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x;
    const int gs = E / n_groups;

    float ss = 0.0f;
    for (int j = threadIdx.x * 8; j < d; j += SEL_WARPS * 32 * 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(u + (size_t)t * d + j);
        *reinterpret_cast<uint4*>(ut + j) = v;
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float lo = bf16_bits_to_float(static_cast<uint16_t>(w[i] & 0xFFFFu));
            const float hi = bf16_bits_to_float(static_cast<uint16_t>(w[i] >> 16));
            ss = fmaf(lo, lo, fmaf(hi, hi, ss));
        }
    }
    for (int e = threadIdx.x; e < NV * 32; e += SEL_WARPS * 32) zex[e] = __int_as_float(0x7fc00000);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0) red[warp] = ss;
    __syncthreads();

    // the best `n` values of group g in arr (NaN entries skipped), summed largest
    // first; also returns the n-th largest
    auto group_best = [&](const float* arr, int g, int n, float& nth) -> float {
        float acc = 0.0f, prev = FLT_MAX;
        int prev_e = -1;
        nth = -FLT_MAX;
        for (int k = 0; k < n; ++k) {
            float best = -FLT_MAX;
            int be = -1;
            for (int e = g * gs; e < (g + 1) * gs; ++e) {
                const float v = arr[e];
                if (v != v) continue;
                // strictly after (prev, prev_e) in the order (value desc, index asc)
                const bool after = v < prev || (v == prev && e > prev_e);
                if (after && (be < 0 || v > best)) { best = v; be = e; }
            }
            if (be < 0) break;
            acc += best;
            nth = best;
            prev = best;
            prev_e = be;
        }
        return acc;
    };

    bool possible = false;
    float za[NV], lo[NV], hi[NV];
    if (warp == 0) {
        ss = 0.0f;
#pragma unroll
        for (int w = 0; w < SEL_WARPS; ++w) ss += red[w];
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int e = j * 32 + lane;
            if (e < E) {
                float l = 0.0f;
                for (int s = 0; s < split; ++s) l += part[((size_t)s * T + t) * E + e];
                za[j] = sigmoid(l) + bias[e];
                const float eps = 0.25f * GAMMA * sqrtf(ss) * norms[e] + 1e-6f +
                                  0x1p-22f * (fabsf(za[j]) + 1.0f);
                lo[j] = za[j] - eps;
                hi[j] = za[j] + eps;
                zlo[e] = lo[j];
                zhi[e] = hi[j];
            } else {
                za[j] = lo[j] = hi[j] = -FLT_MAX;
            }
        }
        __syncwarp();
        // round A: bounds of the group scores, the groups that could reach the cut
        float lg = -FLT_MAX, Lg = -FLT_MAX, ug = -FLT_MAX, dummy;
        if (lane < n_groups) {
            lg = group_best(zlo, lane, group_topk, Lg);
            ug = group_best(zhi, lane, group_topk, dummy);
            ug += 0x1p-22f * group_topk * (fabsf(ug) + 1.0f);     // float32 rounding of the sums
            lg -= 0x1p-22f * group_topk * (fabsf(lg) + 1.0f);
        }
        float lgv[1] = {lg};
        const float LM = kth_largest(lgv, n_groups, topk_groups, lane);
        possible = lane < n_groups && ug >= LM - 2e-6f;
        // in a possible group, the experts that could be among its best group_topk
        int cnt = 0;
        if (possible)
            for (int e = lane * gs; e < (lane + 1) * gs; ++e)
                cnt += zhi[e] >= Lg;
        int incl = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (total > CAND_CAP) {
            // too many: every expert is recomputed
            for (int e = lane; e < E; e += 32) work[e] = e;
            if (lane == 0) { n_work = E; all_mode = 1; }
        } else {
            int at = incl - cnt;
            if (possible)
                for (int e = lane * gs; e < (lane + 1) * gs; ++e)
                    if (zhi[e] >= Lg) work[at++] = e;
            if (lane == 0) { n_work = total; all_mode = 0; }
        }
    }
    __syncthreads();
    auto run_work = [&]() {
        const int n = n_work;
        for (int k = warp; k < n; k += SEL_WARPS) {
            const int e = work[k];
            const float l = exact_dot(ut, c + (size_t)e * d, d, lane);
            if (lane == 0) {
                const float sv = sigmoid(l);
                sex[e] = sv;
                zex[e] = sv + bias[e];
            }
        }
    };
    run_work();
    __syncthreads();

    unsigned keptmask = 0;
    if (warp == 0) {
        const bool all = all_mode != 0;
        // exact scores of the groups in question, the kept groups, group near tie
        float gx = -FLT_MAX, dummy;
        if (lane < n_groups && (possible || all)) gx = group_best(zex, lane, group_topk, dummy);
        unsigned taken = 0;
        float gm = -FLT_MAX, gm1 = -FLT_MAX;
        for (int k = 0; k < topk_groups + 1 && k < n_groups; ++k) {
            float bz = (lane < n_groups && !taken) ? gx : -FLT_MAX;
            int be = (lane < n_groups && !taken) ? lane : 0x7fffffff;
            float wz = bz;
            int we = be;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float oz = __shfl_xor_sync(0xffffffffu, wz, off);
                const int oe = __shfl_xor_sync(0xffffffffu, we, off);
                if (better(oz, oe, wz, we)) { wz = oz; we = oe; }
            }
            if (k < topk_groups) {
                if (lane == we) taken = 1;
                keptmask |= 1u << we;
                if (k == topk_groups - 1) gm = wz;
            } else {
                gm1 = wz;
            }
        }
        if (lane == 0) gtie_sh = (topk_groups < n_groups && gm1 != -FLT_MAX && (gm - gm1) < 1e-6f);
        // round B: in the kept groups, every expert whose upper bound reaches the
        // K-th largest lower bound (less the tie band)
        float zk[NV];
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int e = j * 32 + lane;
            zk[j] = (e < E && (keptmask >> (e / gs) & 1u)) ? lo[j] : -FLT_MAX;
        }
        const float LK = kth_largest(zk, E, K, lane);
        unsigned need = 0;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int e = j * 32 + lane;
            const bool in = e < E && (keptmask >> (e / gs) & 1u);
            const bool band = all || hi[j] >= LK - 2e-6f;
            if (in && band && zex[e] != zex[e]) need |= 1u << j;
        }
        int base = 0;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const unsigned m = __ballot_sync(0xffffffffu, (need >> j) & 1u);
            if ((need >> j) & 1u) work[base + __popc(m & ((1u << lane) - 1u))] = j * 32 + lane;
            base += __popc(m);
        }
        if (lane == 0) n_work = base;
    }
    __syncthreads();
    run_work();
    __syncthreads();
    if (warp != 0) return;

    // selection among the kept groups' recomputed experts
    float s[NV], z[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const int e = j * 32 + lane;
        const bool ok = e < E && (keptmask >> (e / gs) & 1u) && zex[e] == zex[e];
        s[j] = ok ? sex[e] : 0.0f;
        z[j] = ok ? zex[e] : -FLT_MAX;
    }
    unsigned taken = 0;
    float my_s = 0.0f, ssum = 0.0f, zsel = 0.0f, zsel1 = -FLT_MAX;
    int my_e = -1;
    for (int k = 0; k < K + 1; ++k) {
        float bz = -FLT_MAX;
        int be = 0x7fffffff, bj = -1;
        float bs = 0.0f;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int e = j * 32 + lane;
            if (z[j] != -FLT_MAX && !(taken >> j & 1u) && better(z[j], e, bz, be)) {
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
        if (we == be && bj >= 0) taken |= 1u << bj;
        if (k < K) {
            ssum += ws;
            if (lane == k) { my_e = we; my_s = ws; }
            if (k == K - 1) zsel = wz;
        } else {
            zsel1 = wz;                                  // -FLT_MAX: nobody left
        }
    }
    if (lane < K) {
        idx[(size_t)t * K + lane] = my_e;
        gate[(size_t)t * K + lane] = __fdiv_rn(my_s, ssum);
        atomicAdd(&counts[my_e], 1);
    }
    if (lane == 0) {
        const bool ktie = zsel1 != -FLT_MAX && (zsel - zsel1) < 1e-6f;
        tie[t] = (ktie || gtie_sh) ? 1 : 0;
    }
}

template <int NV>
int launch_select_grouped(const uint16_t* u, const float* c, const float* bias, const float* part,
                          int split, int T, int d, int E, int K, int n_groups, int topk_groups,
                          int group_topk, const float* norms, int32_t* idx, float* gate,
                          uint8_t* tie, int32_t* counts, cudaStream_t st) {
    const size_t smem = (size_t)d * 2 + (size_t)NV * 32 * 20;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(select_refine_grouped_kernel<NV>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return launch_pdl(select_refine_grouped_kernel<NV>, dim3(T), dim3(SEL_WARPS * 32), smem, st, u, c,
                      bias, part, split, T, d, E, K, n_groups, topk_groups, group_topk, norms, idx,
                      gate, tie, counts);
}

// Screen, exact recomputation by expert, selection (the workspace's candidate
// lists, exact logits and expert buckets; see route_ws).
template <int NV>
int launch_select2(const uint16_t* u, const float* c, const float* bias, const float* part,
                   int split, int T, int d, int E, int K, const float* norms, int32_t* idx,
                   float* gate, uint8_t* tie, int32_t* counts, void* ws, cudaStream_t st) {
    static int sm_count = 0;
    if (sm_count == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (sm_count <= 0) sm_count = 148;
    }
    const RouteWs W = route_ws(T, d, E);
    char* base = static_cast<char*>(ws);
    int32_t* cand_n = reinterpret_cast<int32_t*>(base + W.cand_n);
    int32_t* cand_e = reinterpret_cast<int32_t*>(base + W.cand_e);
    float* exact = reinterpret_cast<float*>(base + W.exact);
    int32_t* bucket_cnt = reinterpret_cast<int32_t*>(base + W.bucket_cnt);
    int32_t* bucket = reinterpret_cast<int32_t*>(base + W.bucket);
    // (bucket_cnt was zeroed by the split kernel of this call)
    const int tb = (T + SCR_WARPS - 1) / SCR_WARPS;
    int rc = launch_pdl(screen_kernel<NV>, dim3(tb), dim3(SCR_WARPS * 32), 0, st, u, bias, part,
                        split, T, d, E, K, norms, cand_n, cand_e, bucket_cnt, bucket);
    if (rc) return rc;
    const size_t smem = sizeof(float) * (size_t)d + sizeof(int) * (size_t)(E + 1);
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(
            exact_pairs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    // one wave of resident blocks (every block then holds a similar run of pairs)
    static int per_sm = 0;
    static size_t per_sm_smem = 0;
    if (per_sm == 0 || per_sm_smem != smem) {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, exact_pairs_kernel, EX_WARPS * 32, smem) !=
                cudaSuccess || b < 1)
            b = 1;
        per_sm = b;
        per_sm_smem = smem;
    }
    const long long pairs_max = (long long)T * (E < CAND_CAP ? E : CAND_CAP);
    const long long want = (long long)per_sm * sm_count;
    const int grid = (int)(pairs_max < want ? (pairs_max > 0 ? pairs_max : 1) : want);
    if ((rc = launch_pdl(exact_pairs_kernel, dim3(grid), dim3(EX_WARPS * 32), smem, st, u, c, T, d, E,
                         (const int32_t*)bucket_cnt, (const int32_t*)bucket, exact)))
        return rc;
    return launch_pdl(select_exact_kernel<NV>, dim3((T + SEL2_WARPS - 1) / SEL2_WARPS),
                      dim3(SEL2_WARPS * 32), 0, st, u, c, bias, T, d, E, K, (const int32_t*)cand_n,
                      (const int32_t*)cand_e, (const float*)exact, idx, gate, tie, counts);
}

// ------------------------------------------------------------ gate term
// Input gradient through the gates (reading R15): with dg_k = dh_t . y_k (the
// forward's bf16 expert output of slot k), s_k = sigmoid(u_t . e_k) (exact
// logit, as the router) and S = sum_k s_k, the gates g_k = s_k / S give
// dl_k = (dg_k - sum_j g_j dg_j) / S * s_k (1 - s_k), and du_t += sum_k dl_k e_k.
// One block of SEL_WARPS warps per token; the warps share the K slots.
__global__ void __launch_bounds__(SEL_WARPS * 32) gate_term_kernel(
    const uint16_t* __restrict__ u, const uint16_t* __restrict__ dh, const uint16_t* __restrict__ Y,
    const int32_t* __restrict__ inv_row, const int32_t* __restrict__ idx,
    const float* __restrict__ gate, const float* __restrict__ c, int T, int d, int K, int M,
    float* __restrict__ du, int32_t* status) {
    extern __shared__ __align__(16) uint16_t gt_u[];
    __shared__ float dg_s[kMaxTopK], s_s[kMaxTopK], dl_s[kMaxTopK];
    __shared__ int e_s[kMaxTopK];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x;
    for (int j = threadIdx.x * 8; j < d; j += SEL_WARPS * 32 * 8)
        *reinterpret_cast<uint4*>(gt_u + j) = *reinterpret_cast<const uint4*>(u + (size_t)t * d + j);
    __syncthreads();
    for (int k = warp; k < K; k += SEL_WARPS) {
        const int e = idx[(size_t)t * K + k];
        int row = inv_row[(size_t)t * K + k];
        if (row < 0 || row >= M) {
            if (lane == 0) flag_status(status, MOE_ERR_BAD_INDEX);
            row = 0;
        }
        float acc = 0.0f;
        for (int j = lane * 8; j < d; j += 256) {
            const uint4 a = *reinterpret_cast<const uint4*>(dh + (size_t)t * d + j);
            const uint4 b = *reinterpret_cast<const uint4*>(Y + (size_t)row * d + j);
            const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc = fmaf(bf16_bits_to_float(static_cast<uint16_t>(wa[i] & 0xFFFFu)),
                           bf16_bits_to_float(static_cast<uint16_t>(wb[i] & 0xFFFFu)), acc);
                acc = fmaf(bf16_bits_to_float(static_cast<uint16_t>(wa[i] >> 16)),
                           bf16_bits_to_float(static_cast<uint16_t>(wb[i] >> 16)), acc);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        const float l = exact_dot(gt_u, c + (size_t)e * d, d, lane);
        if (lane == 0) {
            dg_s[k] = acc;
            s_s[k] = sigmoid(l);
            e_s[k] = e;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float S = 0.0f, gdg = 0.0f;
        for (int k = 0; k < K; ++k) {
            S += s_s[k];
            gdg = fmaf(gate[(size_t)t * K + k], dg_s[k], gdg);
        }
        for (int k = 0; k < K; ++k) dl_s[k] = __fdiv_rn(dg_s[k] - gdg, S) * s_s[k] * (1.0f - s_s[k]);
    }
    __syncthreads();
    for (int j = threadIdx.x; j < d; j += SEL_WARPS * 32) {
        float v = 0.0f;
        for (int k = 0; k < K; ++k) v = fmaf(dl_s[k], c[(size_t)e_s[k] * d + j], v);
        du[(size_t)t * d + j] += v;
    }
}

__global__ void sum_partials_kernel(const float* __restrict__ part, int split, size_t n,
                                    float* __restrict__ out) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        float v = 0.0f;
        for (int s = 0; s < split; ++s) v += part[s * n + i];
        out[i] = v;
    }
}

// Steps 1 and 2 of the router: the centroid pieces and norms, and the
// partial logit estimates.
int estimate_logits(const uint16_t* u, const float* cent, int T, int d, int E, void* ws,
                    int32_t* status, cudaStream_t st, const float** part_out, int* split_out,
                    const float** norms_out, int32_t* counts = nullptr) {
    const RouteWs W = route_ws(T, d, E);
    char* base = static_cast<char*>(ws);
    float* norms = reinterpret_cast<float*>(base + W.norms);
    uint16_t* hi = reinterpret_cast<uint16_t*>(base + W.hi);
    uint16_t* mid = reinterpret_cast<uint16_t*>(base + W.mid);
    float* part = reinterpret_cast<float*>(base + W.part);
    int rc;
    int32_t* bucket_cnt = counts ? reinterpret_cast<int32_t*>(base + W.bucket_cnt) : nullptr;
    if ((rc = launch_pdl(split_centroids_kernel, dim3(E), dim3(SPLIT_THREADS), 0, st, cent, E, d, hi,
                         mid, norms, counts, bucket_cnt)))
        return rc;
    static bool attr_set = false;
    if (!attr_set) {
        const cudaError_t e = cudaFuncSetAttribute(
            logits_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)RT_SMEM_BYTES);
        if (e != cudaSuccess) return cuda_fail(e);
        attr_set = true;
    }
    CUtensorMap mU, mH, mM;
    if ((rc = make_map_2d(&mU, u, (uint64_t)T, (uint64_t)d, 2, RT_M, RT_K))) return rc;
    if ((rc = make_map_2d(&mH, hi, (uint64_t)E, (uint64_t)d, 2, RT_N, RT_K))) return rc;
    if ((rc = make_map_2d(&mM, mid, (uint64_t)E, (uint64_t)d, 2, RT_N, RT_K))) return rc;
    const dim3 grid((T + RT_M - 1) / RT_M, (E + RT_N - 1) / RT_N, W.split);
    if ((rc = launch_pdl(logits_tc_kernel, grid, dim3(RT_THREADS), RT_SMEM_BYTES, st, mU, mH, mM, T,
                         d, E, W.split, part, status)))
        return rc;
    *part_out = part;
    *split_out = W.split;
    *norms_out = norms;
    return MOE_OK;
}

}  // namespace

size_t route_ws_bytes(int T, int d, int E) { return route_ws(T, d, E).total; }

// Below this many tokens the layer routes with the CUDA-core router (all E
// logits summed exactly, launch_route): the tensor-core screen's fixed costs
// (centroid split, estimate, one refinement block per token) exceed the
// exact sums there (measured on B300, V3 decode shapes: 25-36 us against
// 42-55 us for T <= 128; equal near T = 256).
constexpr int kSmallRouteT = 256;

int launch_route_layer(const uint16_t* u, const float* cent, const float* bias, int T, int d, int E,
                       int K, int32_t* idx, float* gate, uint8_t* tie, int32_t* counts, void* ws,
                       int32_t* status, cudaStream_t st, int n_groups, int topk_groups,
                       int group_topk) {
    const RouteWs w = route_ws(T, d, E);
    if (n_groups == 0 && T > 0 && T < kSmallRouteT && (size_t)T * E * 4 <= (size_t)E * d * 2) {
        // the logits [T, E] and the split partials go where the tensor-core path
        // keeps its centroid pieces and partial estimates
        char* base = static_cast<char*>(ws);
        float* logits = reinterpret_cast<float*>(base + w.hi);
        const size_t part_at = align_up(w.hi + sizeof(float) * (size_t)T * E, 256);
        float* part = reinterpret_cast<float*>(base + part_at);
        const size_t part_floats = (w.total - part_at) / sizeof(float);
        return launch_route(u, cent, bias, T, d, E, K, idx, gate, tie, counts, logits, st, part,
                            part_floats);
    }
    return launch_route_tc(u, cent, bias, T, d, E, K, idx, gate, tie, counts, ws, status, st,
                           n_groups, topk_groups, group_topk);
}

int launch_gate_term(const uint16_t* u, const uint16_t* dh, const uint16_t* Y, const int32_t* inv_row,
                     const int32_t* idx, const float* gate, const float* cent, int T, int d, int K,
                     int M, float* du, int32_t* status, cudaStream_t st) {
    if (T == 0) return MOE_OK;
    const size_t smem = (size_t)d * 2;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(gate_term_kernel,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    gate_term_kernel<<<T, SEL_WARPS * 32, smem, st>>>(u, dh, Y, inv_row, idx, gate, cent, T, d, K, M,
                                                      du, status);
    return check_launch();
}

int launch_route_estimate(const uint16_t* u, const float* cent, int T, int d, int E, float* out,
                          float* norms_out, void* ws, int32_t* status, cudaStream_t st) {
    if (T == 0) return MOE_OK;
    const float* part;
    const float* norms;
    int split, rc;
    if ((rc = estimate_logits(u, cent, T, d, E, ws, status, st, &part, &split, &norms))) return rc;
    const size_t n = (size_t)T * E;
    sum_partials_kernel<<<(int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096), 256, 0, st>>>(
        part, split, n, out);
    if ((rc = check_launch())) return rc;
    const cudaError_t e = cudaMemcpyAsync(norms_out, norms, sizeof(float) * (size_t)E,
                                          cudaMemcpyDeviceToDevice, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

int launch_route_tc(const uint16_t* u, const float* cent, const float* bias, int T, int d, int E,
                    int K, int32_t* idx, float* gate, uint8_t* tie, int32_t* counts, void* ws,
                    int32_t* status, cudaStream_t st, int n_groups, int topk_groups,
                    int group_topk) {
    if (T == 0) {
        const cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)E, st);
        return e == cudaSuccess ? MOE_OK : cuda_fail(e);
    }
    const float* part;
    const float* norms;
    int split, rc;
    if ((rc = estimate_logits(u, cent, T, d, E, ws, status, st, &part, &split, &norms, counts))) return rc;
    const int nv = (E + 31) / 32;
    if (n_groups > 0) {
#define MOE_GROUPED(N)                                                                          \
    return launch_select_grouped<N>(u, cent, bias, part, split, T, d, E, K, n_groups, topk_groups, \
                                    group_topk, norms, idx, gate, tie, counts, st)
        if (nv <= 1) MOE_GROUPED(1);
        if (nv <= 2) MOE_GROUPED(2);
        if (nv <= 4) MOE_GROUPED(4);
        if (nv <= 8) MOE_GROUPED(8);
        if (nv <= 16) MOE_GROUPED(16);
        MOE_GROUPED(32);
#undef MOE_GROUPED
    }
#define MOE_SELECT(N) \
    return launch_select2<N>(u, cent, bias, part, split, T, d, E, K, norms, idx, gate, tie, counts, ws, st)
    if (nv <= 1) MOE_SELECT(1);
    if (nv <= 2) MOE_SELECT(2);
    if (nv <= 4) MOE_SELECT(4);
    if (nv <= 8) MOE_SELECT(8);
    if (nv <= 16) MOE_SELECT(16);
    MOE_SELECT(32);
#undef MOE_SELECT
}

}  // namespace moe
