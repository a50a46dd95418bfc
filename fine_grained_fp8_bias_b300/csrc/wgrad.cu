// Weight gradients of the expert FFNs: the 128x1 re-quantisation of the FP8
// tensors the layer holds, and the token-contracted FP8 GEMM, on sm_103a.
//
// The pages keep FP8 activations in storage and master weights and their
// gradients in 16/32 bits ("DeepSeek V3技術報告", FP8 資料格式訓練;
// "官方揭秘DeepSeek-V3模型训练全流程" §4.3), and ask for transposed GEMMs in
// hardware (same page, hardware suggestions): the tensors the forward holds
// in 1x128 tiles along features are contracted over tokens by the weight
// gradient.  Reading: each such tensor is dequantised (x = dec(q) * s, a
// float32 product), transposed and re-quantised in 128x1 tiles -- 128
// consecutive dispatch rows of one group by one column, the group's last
// block ragged, a block never spanning two groups -- with the forward's
// amax / 448 rule.  Then, per group g and slab kb of its rows,
//     dW[n, m] = sum_kb fma(p_kb[n, m], sA[kb, n] * sB[kb, m], .)
// in float32, p_kb the tensor-core sum of the slab.
//
// Layouts.  A transposed operand of C columns is [C, ld] codes: group g's
// rows occupy columns 128 pb[g] .. 128 pb[g+1] - 1, where pb is the prefix sum
// of ceil(rows_g / 128) (codes past a group's last row are 0); its scales are
// [ld / 128, C] (slab-major, the C values of one slab contiguous).
//
// GEMM kernel shape (one persistent CTA per SM, 384 threads): warp 0 TMA
// producer (A box 128 x 128, B boxes 2 x 128 x 128 per slab, 3-stage ring);
// warp 1 TMEM allocator and MMA issuer (tcgen05.mma.kind::f8f6f4, M = 128,
// N = 256, four K = 32 steps per slab, two TMEM buffers); warp 2 scale loader
// (the slab's 128 row scales and 256 column scales into a shared-memory ring);
// warps 4..11 epilogue (TMEM lane quarter = warp % 4, column half = warpgroup)
// promoting every slab into float32 registers, then writing the 128 x 256
// float32 tile with TMA stores through two 4 KB swizzled staging buffers per
// warp.  Tiles (group, 128-row block of the output, 256-column block) are
// claimed through an atomic counter, group-major, so CTAs working at the same
// time share one group's operands through L2.  Every wait is bounded as in
// the forward GEMM.
#include <cuda.h>
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {
using namespace tc;

// ------------------------------------------------------- re-quantisation
// Two E4M3 codes (lo = low byte) to float32, exactly (E4M3 values are exact
// in f16 and f32).
__device__ __forceinline__ float2 e4m3x2_to_f32(uint16_t v) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
    float lo, hi;
    asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"(static_cast<uint16_t>(h2 & 0xFFFFu)));
    asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"(static_cast<uint16_t>(h2 >> 16)));
    return make_float2(lo, hi);
}

// pb[g] for g = 0..G (padded slab offsets) from the row offsets go, by one
// warp; false (and MOE_ERR_BAD_INDEX) when go is not a non-decreasing list in
// [0, M].
__device__ bool warp_slab_offsets(const int32_t* go, int G, int M, int* pb, int32_t* status) {
    const int lane = threadIdx.x & 31;
    int carry = 0;
    bool bad = false;
    for (int base = 0; base <= G; base += 32) {
        const int g = base + lane;
        int v = 0;
        if (g < G) {
            const int a = go[g], b = go[g + 1];
            if (a < 0 || b < a || b > M) bad = true;
            v = (max(0, b - a) + 127) / 128;
        }
        int incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (g <= G) pb[g] = carry + incl - v;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (bad && lane == 0) flag_status(status, MOE_ERR_BAD_INDEX);
    return !bad;
}

// Shared memory of the re-quantisation kernel (dynamic: above 48 KB).
struct RqSmem {
    uint8_t tile[2][128][128];          // double-buffered input tile [row][column]
    uint32_t tq[128][33];               // output tile [column][row / 4], 4 codes a word
    float part[8][128];                 // column amax of each warp's 16 rows
    int pb[kMaxGroups + 1];
    float rs[2][128];                   // row scales of each buffer
    int ok;
};

// x / scale correctly rounded, from r = RN(1 / scale), with no division:
// y = RN(x r) is within 2 ulps of the quotient; one correction step
// q1 = RN(y + RN(x - scale y) r) makes it faithful (within 1 ulp), and a
// second step from a faithful quotient with the correctly rounded reciprocal
// gives the correctly rounded quotient (Markstein, IBM J. Res. Dev. 34(1),
// 1990; the residual x - scale q1 is exact in one FMA).  The correction sums
// turn a -0 quotient into +0, so the sign is taken from x.  Valid for finite x
// and scale >= 2^-100 (no underflow in the residuals that matters: a quotient
// below 2^-10 encodes to 0 whatever its last bits).
__device__ __forceinline__ float div_rn_rcp(float x, float scale, float r) {
    const float y = x * r;
    const float q1 = fmaf(fmaf(-scale, y, x), r, y);
    const float q2 = fmaf(fmaf(-scale, q1, x), r, q1);
    return copysignf(q2, x);
}

// One block per padded slab j (128 rows of one group) and a stride of
// 128-column blocks: the group lookup is paid once, then the column blocks
// stream through a two-deep cp.async ring (load of block k+1 in flight while
// block k is converted and written).  Thread (warp w, lane l) converts the
// four columns 4l .. 4l + 3 of rows 16 w .. 16 w + 15: one 32-bit shared
// load brings a row's four codes.
__global__ void __launch_bounds__(256, 4) requant_128x1_kernel(const uint8_t* __restrict__ q,
                                                               const float* __restrict__ s, int M,
                                                               int C, const int32_t* __restrict__ go,
                                                               int G, uint8_t* __restrict__ qt,
                                                               float* __restrict__ st, int ld,
                                                               int32_t* status) {
    extern __shared__ __align__(16) uint8_t rq_raw[];
    RqSmem& sm = *reinterpret_cast<RqSmem*>(rq_raw);
    const int tid = threadIdx.x;
    const int j = blockIdx.y;
    const int ncb = C / 128;
    // the group offsets through shared memory (one coalesced read), then the scan
    int* gos = reinterpret_cast<int*>(&sm.tq[0][0]);      // tq is free until the first block
    for (int g = tid; g <= G; g += 256) gos[g] = go[g];
    __syncthreads();
    if (tid < 32) {
        const bool ok = warp_slab_offsets(gos, G, M, sm.pb, status);
        if (tid == 0) sm.ok = ok;
    }
    __syncthreads();
    if (!sm.ok || j >= sm.pb[G]) return;
    if (sm.pb[G] > ld / 128) {               // the padded rows do not fit the output
        if (tid == 0) flag_status(status, MOE_ERR_BAD_INDEX);
        return;
    }
    int lo = 0, hi = G;                      // pb[lo] <= j < pb[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (sm.pb[mid] <= j) lo = mid; else hi = mid;
    }
    const int r0 = gos[lo] + (j - sm.pb[lo]) * 128;
    const int n = min(128, gos[lo + 1] - r0);
    __syncthreads();                         // gos (in tq) is read by all before tq is reused

    // rows r0 .. r0 + n - 1 of column block cb into buffer b; rows past n are zero
    auto stage = [&](int cb, int b) {
        for (int i = tid; i < 128 * 8; i += 256) {
            const int r = i >> 3, c16 = (i & 7) * 16;
            const bool v = r < n;
            cp_async16(&sm.tile[b][r][c16], v ? q + (size_t)(r0 + r) * C + (size_t)cb * 128 + c16 : q,
                       v ? 16u : 0u);
        }
        if (tid < 128) {
            const bool v = tid < n;
            cp_async4(&sm.rs[b][tid], v ? s + (size_t)cb * M + r0 + tid : s, v ? 4u : 0u);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    const int warp = tid >> 5, lane = tid & 31;
    const int c0 = 4 * lane, rw = 16 * warp;
    // x = dec(code) * row scale for row r, columns c0 .. c0 + 3
    auto deq = [&](int b, int r, float (&x)[4]) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(&sm.tile[b][r][c0]);
        const float2 f0 = e4m3x2_to_f32(static_cast<uint16_t>(w & 0xFFFFu));
        const float2 f1 = e4m3x2_to_f32(static_cast<uint16_t>(w >> 16));
        const float sr = sm.rs[b][r];
        x[0] = __fmul_rn(f0.x, sr);
        x[1] = __fmul_rn(f0.y, sr);
        x[2] = __fmul_rn(f1.x, sr);
        x[3] = __fmul_rn(f1.y, sr);
    };
    int cb = blockIdx.x;
    if (cb < ncb) stage(cb, 0);
    for (int k = 0; cb < ncb; ++k, cb += gridDim.x) {
        const int b = k & 1;
        const bool more = cb + (int)gridDim.x < ncb;
        if (more) stage(cb + gridDim.x, b ^ 1);
        if (more) asm volatile("cp.async.wait_group 1;" ::: "memory");
        else asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        // pass 1: column amax over this warp's 16 rows, then over the 8 warps
        float am[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
            float x[4];
            deq(b, rw + i, x);
#pragma unroll
            for (int t = 0; t < 4; ++t) am[t] = fmaxf(am[t], fabsf(x[t]));
        }
        *reinterpret_cast<float4*>(&sm.part[warp][c0]) = make_float4(am[0], am[1], am[2], am[3]);
        __syncthreads();
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const float4 v = *reinterpret_cast<const float4*>(&sm.part[w][c0]);
            am[0] = fmaxf(am[0], v.x);
            am[1] = fmaxf(am[1], v.y);
            am[2] = fmaxf(am[2], v.z);
            am[3] = fmaxf(am[3], v.w);
        }
        float sc[4], rc[4];
        bool all_fast = true;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            sc[t] = tile_scale(am[t]);
            rc[t] = __frcp_rn(sc[t]);
            all_fast = all_fast && sc[t] >= 0x1p-100f;
        }
        if (warp == 0)
            *reinterpret_cast<float4*>(st + (size_t)j * C + (size_t)cb * 128 + c0) =
                make_float4(sc[0], sc[1], sc[2], sc[3]);
        // pass 2: four rows at a time; column t's four codes make one word of tq
        // (an all-zero column gets code 0); IEEE division for scales near underflow
        auto pass2 = [&](auto div) {
#pragma unroll 1
            for (int i = 0; i < 16; i += 4) {
                float x[4][4];
#pragma unroll
                for (int u = 0; u < 4; ++u) deq(b, rw + i + u, x[u]);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    float y[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) y[u] = div(x[u][t], t);
                    const uint32_t word = static_cast<uint32_t>(e4m3x2(y[0], y[1])) |
                                          (static_cast<uint32_t>(e4m3x2(y[2], y[3])) << 16);
                    sm.tq[c0 + t][(rw + i) >> 2] = am[t] != 0.0f ? word : 0u;
                }
            }
        };
        if (all_fast)
            pass2([&](float v, int t) { return div_rn_rcp(v, sc[t], rc[t]); });
        else
            pass2([&](float v, int t) { return __fdiv_rn(v, sc[t]); });
        __syncthreads();
        // row cc of the output tile: 128 codes, one coalesced 128-byte write per warp
        for (int cc = warp; cc < 128; cc += 8)
            *reinterpret_cast<uint32_t*>(qt + (size_t)(cb * 128 + cc) * ld + (size_t)j * 128 + lane * 4) =
                sm.tq[cc][lane];
        __syncthreads();                     // tq, part and buffer b are reused next round
    }
}

// -------------------------------------------------------------- the GEMM
constexpr int BM = 128;
constexpr int BK = 128;
constexpr int BN = 256;
constexpr int STAGES = 3;
constexpr int SMEM_A = BM * BK;                 // 16 KB
constexpr int SMEM_B = BN * BK;                 // 32 KB
constexpr int SMEM_STAGE = SMEM_A + SMEM_B;
constexpr int NUM_EPI_WARPS = 8;
constexpr int EPI_WARP0 = 4;
constexpr int NUM_THREADS = 128 + 32 * NUM_EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;
constexpr int SCALE_SLOTS = 6;
constexpr int SCALE_LAG = 2;
constexpr int TILE_SLOTS = 4;
constexpr int TILE_READERS = 2 + NUM_EPI_WARPS;
constexpr int OUT_CHUNK = 32 * 32 * 4;          // one 32 x 32 float32 staging buffer
constexpr int SMEM_OUT = NUM_EPI_WARPS * 2 * OUT_CHUNK;
constexpr int LAUNCH_REGS = 168;
constexpr int CTRL_REGS = 40;
constexpr int EPI_REGS = 232;
static_assert(128 * CTRL_REGS + 256 * EPI_REGS <= NUM_THREADS * LAUNCH_REGS, "register split");

struct alignas(16) ScaleSlot {
    float sa[BM];                               // scale of each output row (A operand row)
    float sb[BN];                               // scale of each output column (B operand row)
};

struct alignas(16) Ctl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t epi_done;
    uint64_t sfull[SCALE_SLOTS];
    uint64_t sempty[SCALE_SLOTS];
    uint64_t tile_full[TILE_SLOTS];
    uint64_t tile_empty[TILE_SLOTS];
    int tile_ring[TILE_SLOTS];
    uint32_t tmem_base;
    int abort;
    int total_tiles;
    int ok;
    ScaleSlot scales[SCALE_SLOTS];
    int pb[kMaxGroups + 1];                     // padded slab offset of each group
};

constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * SMEM_STAGE + SMEM_OUT + sizeof(Ctl);
static_assert(SMEM_BYTES <= 232448, "shared memory");

struct Params {
    int Na, Nb, G, split;
    int kb_cap;                                 // slabs the operands hold (ld / 128)
    const float* sa;                            // [ld / 128, Na]
    const float* sb;                            // [ld / 128, Nb]
    int32_t* status;
    int* counter;
};

struct WTile {
    int g, rt, ct;
};
__device__ __forceinline__ WTile wtile(int tile, int rtiles, int ctiles) {
    const int per = rtiles * ctiles;
    const int g = tile / per, local = tile - g * per;
    return WTile{g, local / ctiles, local % ctiles};
}

__device__ __forceinline__ bool take_tile(Ctl* ctl, uint32_t& tpos, int& tile, int32_t* status) {
    const int slot = tpos % TILE_SLOTS;
    if (!mbar_wait(&ctl->tile_full[slot], (tpos / TILE_SLOTS) & 1, &ctl->abort, status)) return false;
    tile = ctl->tile_ring[slot];
    mbar_arrive(&ctl->tile_empty[slot]);
    ++tpos;
    return true;
}
__device__ __forceinline__ bool warp_take_tile(Ctl* ctl, uint32_t& tpos, int& tile, int32_t* status) {
    const int slot = tpos % TILE_SLOTS;
    if (!warp_wait(&ctl->tile_full[slot], (tpos / TILE_SLOTS) & 1, &ctl->abort, status)) return false;
    tile = ctl->tile_ring[slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&ctl->tile_empty[slot]);
    ++tpos;
    return true;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    wgrad_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmO0, const __grid_constant__ CUtensorMap tmO1,
                      const int32_t* __restrict__ go, const Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* out_stage = smem + (size_t)STAGES * SMEM_STAGE;
    Ctl* ctl = reinterpret_cast<Ctl*>(out_stage + SMEM_OUT);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int RT = p.Na / BM;
    const int CT = (p.Nb + BN - 1) / BN;

    if (warp == 0) {
        bool ok = warp_slab_offsets(go, p.G, 0x7fffffff, ctl->pb, p.status);
        if (ok && ctl->pb[p.G] > p.kb_cap) {     // more slabs than the operands hold
            ok = false;
            if (lane == 0) flag_status(p.status, MOE_ERR_BAD_INDEX);
        }
        if (lane == 0) {
            ctl->ok = ok;
            ctl->total_tiles = ok ? p.G * RT * CT : 0;
            ctl->abort = 0;
            for (int s = 0; s < STAGES; ++s) {
                mbar_init(&ctl->full[s], 1);
                mbar_init(&ctl->empty[s], 1);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(&ctl->tfull[b], 1);
                mbar_init(&ctl->tempty[b], NUM_EPI_WARPS);
            }
            for (int s = 0; s < SCALE_SLOTS; ++s) {
                mbar_init(&ctl->sfull[s], 32);
                mbar_init(&ctl->sempty[s], NUM_EPI_WARPS);
            }
            for (int s = 0; s < TILE_SLOTS; ++s) {
                mbar_init(&ctl->tile_full[s], 1);
                mbar_init(&ctl->tile_empty[s], TILE_READERS);
            }
            mbar_init(&ctl->epi_done, NUM_EPI_WARPS);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            tma_prefetch_desc(&tmO0);
            if (p.split < p.Na) tma_prefetch_desc(&tmO1);
        }
    } else if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&ctl->tmem_base)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const int total_tiles = ctl->total_tiles;

    if (warp < EPI_WARP0) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(CTRL_REGS));
      // (role code of warpgroup 0 below is indented one level less than its scope)
      if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            uint32_t it = 0, tpos = 0;
            int tile = -1;
            while (true) {
                int next = p.counter ? atomicAdd(p.counter, 1)
                                     : (tile < 0 ? (int)blockIdx.x : tile + (int)gridDim.x);
                if (next >= total_tiles) next = -1;
                const int slot = tpos % TILE_SLOTS;
                if (!mbar_wait(&ctl->tile_empty[slot], ((tpos / TILE_SLOTS) & 1) ^ 1, &ctl->abort,
                               p.status))
                    break;
                ctl->tile_ring[slot] = next;
                mbar_arrive(&ctl->tile_full[slot]);
                ++tpos;
                if (next < 0) break;
                tile = next;
                const WTile tl = wtile(tile, RT, CT);
                const bool has_b1 = tl.ct * BN + 128 < p.Nb;
                const uint32_t bytes = SMEM_A + 128 * BK * (has_b1 ? 2 : 1);
                bool ok = true;
                for (int kb = ctl->pb[tl.g]; kb < ctl->pb[tl.g + 1]; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (!mbar_wait(&ctl->empty[s], ((it / STAGES) & 1) ^ 1, &ctl->abort, p.status)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sA = smem + (size_t)s * SMEM_STAGE;
                    uint8_t* sB = sA + SMEM_A;
                    mbar_expect_tx(&ctl->full[s], bytes);
                    tma_load_2d(sA, &tmA, &ctl->full[s], kb * BK, tl.rt * BM);
                    tma_load_2d(sB, &tmB, &ctl->full[s], kb * BK, tl.ct * BN);
                    if (has_b1) tma_load_2d(sB + 128 * BK, &tmB, &ctl->full[s], kb * BK, tl.ct * BN + 128);
                }
                if (!ok) break;
            }
            const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0;
            for (uint32_t j = first; j < it; ++j) mbar_drain(&ctl->full[j % STAGES], (j / STAGES) & 1);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3(BM, BN);
            uint32_t it = 0, tpos = 0;
            bool ok = true;
            int tile;
            while (ok) {
                if (!take_tile(ctl, tpos, tile, p.status)) break;
                if (tile < 0) break;
                const WTile tl = wtile(tile, RT, CT);
                for (int kb = ctl->pb[tl.g]; kb < ctl->pb[tl.g + 1]; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t buf = it & 1;
                    if (!mbar_wait(&ctl->tempty[buf], ((it >> 1) & 1) ^ 1, &ctl->abort, p.status)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait(&ctl->full[s], (it / STAGES) & 1, &ctl->abort, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(smem + (size_t)s * SMEM_STAGE);
                    const uint32_t b0 = a0 + SMEM_A;
                    const uint32_t d_tmem = tmem_base + buf * BN;
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        mma_e4m3(d_tmem, sdesc_sw128(a0 + k * 32), sdesc_sw128(b0 + k * 32), idesc,
                                 k > 0 ? 1u : 0u);
                    mma_commit(&ctl->empty[s]);
                    mma_commit(&ctl->tfull[buf]);
                }
            }
            if (it > 0) mbar_drain(&ctl->tfull[(it - 1) & 1], ((it - 1) >> 1) & 1);
            mbar_drain(&ctl->epi_done, 0, 3 * WAIT_CYCLES);
        }
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(TMEM_COLS));
    } else if (warp == 2) {
        // ================= scale loader =================
        uint32_t it = 0, tpos = 0;
        bool ok = true;
        int tile;
        while (ok) {
            if (!warp_take_tile(ctl, tpos, tile, p.status)) { ok = false; break; }
            if (tile < 0) break;
            const WTile tl = wtile(tile, RT, CT);
            for (int kb = ctl->pb[tl.g]; kb < ctl->pb[tl.g + 1]; ++kb, ++it) {
                const int slot = it % SCALE_SLOTS;
                bool got = true;
                if (lane == 0)
                    got = mbar_wait(&ctl->sempty[slot], ((it / SCALE_SLOTS) & 1) ^ 1, &ctl->abort, p.status);
                if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) { ok = false; break; }
                ScaleSlot& sl = ctl->scales[slot];
                cp_async16(&sl.sa[lane * 4], p.sa + (size_t)kb * p.Na + tl.rt * BM + lane * 4, 16u);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int col = tl.ct * BN + h * 128 + lane * 4;
                    const bool v = col < p.Nb;
                    cp_async16(&sl.sb[h * 128 + lane * 4], v ? p.sb + (size_t)kb * p.Nb + col : p.sb,
                               v ? 16u : 0u);
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
                if (it >= (uint32_t)SCALE_LAG) {
                    asm volatile("cp.async.wait_group %0;" ::"n"(SCALE_LAG) : "memory");
                    mbar_arrive(&ctl->sfull[(it - SCALE_LAG) % SCALE_SLOTS]);
                }
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (ok)
            for (uint32_t j = it > (uint32_t)SCALE_LAG ? it - SCALE_LAG : 0; j < it; ++j)
                mbar_arrive(&ctl->sfull[j % SCALE_SLOTS]);
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(EPI_REGS));
        // ================= epilogue =================
        const int ew = warp - EPI_WARP0;
        const int wg = ew >> 2;                   // column half
        const int quarter = warp & 3;             // TMEM lane quarter
        const int row = quarter * 32 + lane;      // row within the tile
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        uint8_t* stage0 = out_stage + (size_t)ew * 2 * OUT_CHUNK;
        uint32_t it = 0, tpos = 0, nstore = 0;
        bool ok = true;
        int tile;
        while (ok) {
            if (!warp_take_tile(ctl, tpos, tile, p.status)) { ok = false; break; }
            if (tile < 0) break;
            const WTile tl = wtile(tile, RT, CT);
            const int nkb = ctl->pb[tl.g + 1] - ctl->pb[tl.g];
            const int col0 = tl.ct * BN + wg * 128;      // first output column of this thread
            const bool cols_valid = col0 < p.Nb;
            float acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
            for (int k = 0; k < nkb; ++k, ++it) {
                const int slot = it % SCALE_SLOTS;
                const uint32_t buf = it & 1;
                if (!warp_wait(&ctl->sfull[slot], (it / SCALE_SLOTS) & 1, &ctl->abort, p.status) ||
                    !warp_wait(&ctl->tfull[buf], (it >> 1) & 1, &ctl->abort, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (cols_valid) {
                    const ScaleSlot& sl = ctl->scales[slot];
                    const float sa = sl.sa[row];
                    const float* sb = sl.sb + wg * 128;
                    const uint32_t tbase = tmem_base + lane_addr + buf * BN + wg * 128;
                    uint32_t a[32], b[32];
                    tmem_ld32_nowait(tbase, a);
                    tmem_ld_wait(a);
                    tmem_ld32_nowait(tbase + 32, b);
                    fma2_rowcol<32>(acc, a, sa, sb);
                    tmem_ld_wait(b);
                    tmem_ld32_nowait(tbase + 64, a);
                    fma2_rowcol<32>(acc + 32, b, sa, sb + 32);
                    tmem_ld_wait(a);
                    tmem_ld32_nowait(tbase + 96, b);
                    fma2_rowcol<32>(acc + 64, a, sa, sb + 64);
                    tmem_ld_wait(b);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->tempty[buf]);
                    fma2_rowcol<32>(acc + 96, b, sa, sb + 96);
                } else {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->tempty[buf]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->sempty[slot]);
            }
            if (!ok) break;
            if (!cols_valid) continue;
            // ---- store: four 32 x 32 chunks through the two staging buffers
            const bool second = tl.rt * BM >= p.split;
            const CUtensorMap* map = second ? &tmO1 : &tmO0;
            const int y = second ? tl.g * (p.Na - p.split) + tl.rt * BM - p.split + quarter * 32
                                 : tl.g * p.split + tl.rt * BM + quarter * 32;
#pragma unroll
            for (int q = 0; q < 4; ++q, ++nstore) {
                uint8_t* buf = stage0 + (nstore & 1) * OUT_CHUNK;
                if (lane == 0) bulk_wait_read_1();      // this buffer's previous store has read it
                __syncwarp();
                // row `lane`, 16-byte piece jj at the 128-byte-swizzled position
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const float* v = acc + q * 32 + jj * 4;
                    *reinterpret_cast<float4*>(buf + lane * 128 + ((jj ^ (lane & 7)) << 4)) =
                        make_float4(v[0], v[1], v[2], v[3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(map, buf, col0 + q * 32, y);
                    bulk_commit();
                }
            }
        }
        if (lane == 0) bulk_wait_all();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->epi_done);
    }
}

}  // namespace

int launch_requant_128x1(const uint8_t* q, const float* s, int M, int C, const int32_t* go, int G,
                         uint8_t* qt, float* st, int ld, int32_t* status, cudaStream_t stream) {
    if (M == 0 || G == 0 || C == 0) return MOE_OK;
    const long long slabs = ((long long)M + 127LL * G) / 128 + 1;
    if (slabs > 65535) return MOE_ERR_UNSUPPORTED_SHAPE;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(requant_128x1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(RqSmem));
    });
    // about four blocks per column block stride: enough slabs x strides to fill
    // the SMs while each block amortises its group lookup over several blocks
    const int ncb = C / 128;
    const int stride = ncb < 8 ? ncb : 8;
    requant_128x1_kernel<<<dim3(stride, (unsigned)slabs), 256, sizeof(RqSmem), stream>>>(
        q, s, M, C, go, G, qt, st, ld, status);
    return check_launch();
}

int launch_wgrad_gemm(const uint8_t* At, const float* sAt, int Na, const uint8_t* Bt,
                      const float* sBt, int Nb, int ld, const int32_t* go, int G, float* out0,
                      float* out1, int split, int32_t* status, cudaStream_t st) {
    if (G == 0) return MOE_OK;
    static int sm_count = 0, num_regs = 0;
    static std::once_flag once;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    std::call_once(once, [&] {
        cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
        cudaFuncSetAttribute(wgrad_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES);
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, wgrad_gemm_kernel) == cudaSuccess) num_regs = fa.numRegs;
    });
    if (sm_count <= 0) return cuda_fail(cudaErrorInvalidDevice);
    if (num_regs != LAUNCH_REGS) return cuda_fail(cudaErrorInvalidConfiguration);
    CUtensorMap mA, mB, mO0, mO1;
    int rc = make_map_2d(&mA, At, (uint64_t)Na, (uint64_t)ld, 1, 128, 128);
    if (rc) return rc;
    if ((rc = make_map_2d(&mB, Bt, (uint64_t)Nb, (uint64_t)ld, 1, 128, 128))) return rc;
    if ((rc = make_map_2d(&mO0, out0, (uint64_t)G * split, (uint64_t)Nb, 4, 32, 32))) return rc;
    if (split < Na) {
        if ((rc = make_map_2d(&mO1, out1, (uint64_t)G * (Na - split), (uint64_t)Nb, 4, 32, 32))) return rc;
    } else {
        mO1 = mO0;
    }
    int* counter = status ? status + 1 : nullptr;
    if (counter) {
        const cudaError_t ce = cudaMemsetAsync(counter, 0, sizeof(int), st);
        if (ce != cudaSuccess) return cuda_fail(ce);
    }
    Params p{Na, Nb, G, split, ld / 128, sAt, sBt, status, counter};
    const long long tiles = (long long)G * (Na / BM) * ((Nb + BN - 1) / BN);
    if (tiles > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int grid = (int)(tiles < sm_count ? tiles : sm_count);
    wgrad_gemm_kernel<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(mA, mB, mO0, mO1, go, p);
    return check_launch();
}

}  // namespace moe
