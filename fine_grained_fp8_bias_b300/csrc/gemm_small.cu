// Grouped block-scaled FP8 GEMM for groups with few rows (decode batches),
// on sm_103a tensor cores.
//
// Source: "รายงานเชิงเทคนิคของ DeepSeek-V3" (xyznot.com/th/paper/2412.19437),
// Key ideas, FP8 bullet, and "官方揭秘DeepSeek-V3模型训练全流程"
// (youleyou.com) §4.3: E4M3 operands with one FP32 scale per 1x128
// activation tile and per 128x128 weight block; each N_c = 128 slab of K is
// summed on the tensor core and promoted to FP32:
//     acc = fma(partial, sa[row, kb] * sw[nb, kb], acc).
// Same contract and arithmetic as grouped_gemm_fp8_kernel (gemm_fp8.cu); only
// the tile shape differs.  With a handful of rows per expert, a 128-row tile
// of activations is mostly padding while the weight panel dominates the
// bytes, so here the operands swap places: the tensor core's M side is 128
// rows of one weight block (the "A" operand) and its N side is a chunk of up
// to 32 rows of the group (N = 16 or 32), D[weight row][row] in TMEM.  A stage
// then holds 16 KB (down) or 32 KB (gate + up) of weights and 4 KB of rows,
// so 5 or 9 stages fit and more weight bytes are in flight per SM; the
// per-slab promotion touches 32 or 64 TMEM columns instead of 256.
//
// Tile = (group g, weight tile nt, row chunk c): weight rows nt*128 .. +128
// (GATE_UP: those gate rows and the same up rows, so SiLU(G) * U and the
// 1x128 re-quantisation of h along the intermediate index stay inside the
// tile), group rows c*32 .. +32.  Tiles are claimed from a counter in the
// order group, weight tile, chunk: the chunks of one weight panel run
// together and read it from HBM once.  A group with many rows (a hot expert)
// is split into as many chunk tiles, each on its own CTA.
//
// Kernel shape (one persistent CTA per SM, 256 threads):
//   warp 0      TMA producer (weight block(s) + 16-row boxes of the chunk)
//   warp 1      TMEM allocator and MMA issuer (4 x tcgen05.mma.kind::f8f6f4,
//               M = 128, N = 16 * boxes, K = 32 per slab and weight block)
//   warp 2      scale loader (the chunk's activation scales and the weight
//               block scales of each slab, cp.async into a ring)
//   warp 3      idle
//   warps 4..7  epilogue: thread (warp, lane) owns weight row
//               32 * (warp % 4) + lane and the chunk's up to 32 rows.
// Every wait is bounded as in gemm_fp8.cu.
#include <cuda.h>
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {
using namespace tc;

constexpr int SK = 128;                         // K slab
constexpr int SWR = 128;                        // weight rows per tile (MMA M)
constexpr int STOK = 32;                        // rows per chunk (MMA N at most)
constexpr int SBOX = 16;                        // rows per TMA box of the chunk
constexpr int SMEM_W = SWR * SK;                // 16 KB per weight block
constexpr int SMEM_T = STOK * SK;               // 4 KB of rows
constexpr int S_THREADS = 256;
constexpr int S_EPI0 = 4;                       // first epilogue warp
constexpr int S_EPI_WARPS = 4;
constexpr int S_NBUF = 4;                       // TMEM buffers
constexpr uint32_t S_TMEM_COLS = 256;           // 4 buffers x 64 columns
constexpr int S_SCALE_SLOTS = 8;
constexpr int S_SCALE_LAG = 3;
constexpr int S_TILE_SLOTS = 4;
constexpr int S_TILE_READERS = 2 + S_EPI_WARPS;

template <int MODE>
struct SmallCfg {
    static constexpr int NW = MODE ? 2 : 1;                 // weight blocks per slab
    static constexpr int STAGE = NW * SMEM_W + SMEM_T;      // 36 KB or 20 KB
    static constexpr int STAGES = MODE ? 5 : 9;
};

struct alignas(16) SScaleSlot {
    float sa[STOK];                              // activation scale of each chunk row (0 outside)
    float sw[4];                                 // weight block scale(s) of the slab
};

struct alignas(16) SCtl {
    uint64_t full[9];
    uint64_t empty[9];
    uint64_t tfull[S_NBUF];
    uint64_t tempty[S_NBUF];
    uint64_t xbar;
    uint64_t epi_done;
    uint64_t sfull[S_SCALE_SLOTS];
    uint64_t sempty[S_SCALE_SLOTS];
    uint64_t tile_full[S_TILE_SLOTS];
    uint64_t tile_empty[S_TILE_SLOTS];
    int tile_ring[S_TILE_SLOTS];
    uint32_t tmem_base;
    int abort;
    int total_tiles;
    int pad;
    float amax[2][S_EPI_WARPS][STOK];           // [tile parity][warp][row]
    SScaleSlot scales[S_SCALE_SLOTS];
    int go[kMaxGroups + 1];
    int tile_start[kMaxGroups + 1];
};

template <int MODE>
constexpr size_t small_smem_bytes() {
    return 1024 + (size_t)SmallCfg<MODE>::STAGES * SmallCfg<MODE>::STAGE + sizeof(SCtl);
}

struct SParams {
    int M_total, G, N, Kdim;
    const int32_t* go;
    const float* sa;
    const float* sw0;
    const float* sw1;
    void* out;
    float* out_scales;
    int32_t* status;
    int* counter;
    int f32_group0;                              // DOWN: rows of groups >= f32_group0 go to
    int f32_row0;                                // out2 (float32, row - f32_row0), the others
    float* out2;                                 // to out (bf16)
    long long wait_cycles;                       // limit of every pipeline wait (SM clock cycles)
    int stall;                                   // test switch: the producer issues no loads
};

struct STile {
    int g, nt, c;
};

__device__ __forceinline__ STile s_find_tile(const SCtl* ctl, int G, int NB, int tile) {
    int lo = 0, hi = G;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (ctl->tile_start[mid] <= tile) lo = mid; else hi = mid;
    }
    const int m = max(0, ctl->go[lo + 1] - ctl->go[lo]);
    const int chunks = (m + STOK - 1) / STOK;
    const int local = tile - ctl->tile_start[lo];
    (void)NB;
    return STile{lo, local / chunks, local % chunks};
}

// Correctly rounded x / scale from r = RN(1 / scale) (two Markstein steps), as
// in the large-tile kernel's epilogue.
__device__ __forceinline__ float s_div_rcp(float x, float scale, float r) {
    const float y = x * r;
    const float q1 = fmaf(fmaf(-scale, y, x), r, y);
    return copysignf(fmaf(fmaf(-scale, q1, x), r, q1), x);
}

__device__ __forceinline__ bool s_take_tile(SCtl* ctl, uint32_t& tpos, int& tile, int32_t* status, long long limit) {
    const int slot = tpos % S_TILE_SLOTS;
    if (!mbar_wait(&ctl->tile_full[slot], (tpos / S_TILE_SLOTS) & 1, &ctl->abort, status, limit)) return false;
    tile = ctl->tile_ring[slot];
    mbar_arrive(&ctl->tile_empty[slot]);
    ++tpos;
    return true;
}
__device__ __forceinline__ bool s_warp_take_tile(SCtl* ctl, uint32_t& tpos, int& tile,
                                                 int32_t* status, long long limit) {
    const int slot = tpos % S_TILE_SLOTS;
    if (!warp_wait(&ctl->tile_full[slot], (tpos / S_TILE_SLOTS) & 1, &ctl->abort, status, limit)) return false;
    tile = ctl->tile_ring[slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&ctl->tile_empty[slot]);
    ++tpos;
    return true;
}

// MODE 0: down projection (y float32 or bf16); 1: gate/up + SiLU + 1x128
// re-quantisation.
template <int MODE>
__global__ void __launch_bounds__(S_THREADS, 1)
    grouped_gemm_small_kernel(const __grid_constant__ CUtensorMap tmA,
                              const __grid_constant__ CUtensorMap tmW0,
                              const __grid_constant__ CUtensorMap tmW1, const SParams p) {
    using C = SmallCfg<MODE>;
    constexpr bool gate_up = MODE != 0;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    SCtl* ctl = reinterpret_cast<SCtl*>(smem + (size_t)C::STAGES * C::STAGE);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int NB = p.N / SWR;
    const int KB = p.Kdim / SK;
    const int G = p.G;

    // Barriers, TMEM and the tensor-map prefetch touch only this CTA's own
    // memory: set up before waiting for the kernel this launch depends on.
    if (warp == 0) {
        if (lane == 0) {
            for (int s = 0; s < C::STAGES; ++s) {
                mbar_init(&ctl->full[s], 1);
                mbar_init(&ctl->empty[s], 1);
            }
            for (int b = 0; b < S_NBUF; ++b) {
                mbar_init(&ctl->tfull[b], 1);
                mbar_init(&ctl->tempty[b], S_EPI_WARPS);
            }
            for (int s = 0; s < S_SCALE_SLOTS; ++s) {
                mbar_init(&ctl->sfull[s], 32);
                mbar_init(&ctl->sempty[s], S_EPI_WARPS);
            }
            for (int s = 0; s < S_TILE_SLOTS; ++s) {
                mbar_init(&ctl->tile_full[s], 1);
                mbar_init(&ctl->tile_empty[s], S_TILE_READERS);
            }
            mbar_init(&ctl->xbar, S_EPI_WARPS);
            mbar_init(&ctl->epi_done, S_EPI_WARPS);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmW0);
            if (gate_up) tma_prefetch_desc(&tmW1);
        }
    } else if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&ctl->tmem_base)),
                     "r"(S_TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    griddep_wait();
    griddep_launch();
    // the group offsets (the preceding kernel's output) in one round of loads,
    // then warp 0's scan: tile_start[g] = sum over g' < g of NB * ceil(m_g' / 32)
    for (int g = threadIdx.x; g <= G; g += S_THREADS) ctl->go[g] = p.go[g];
    __syncthreads();
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base <= G; base += 32) {
            const int g = base + lane;
            int v = 0;
            if (g < G) {
                const int m = max(0, ctl->go[g + 1] - ctl->go[g]);
                v = (m + STOK - 1) / STOK * NB;
            }
            int incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            if (g <= G) ctl->tile_start[g] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            ctl->total_tiles = ctl->tile_start[G];
            ctl->abort = 0;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const int total_tiles = ctl->total_tiles;

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            uint32_t it = 0, tpos = 0;
            int tile = -1;
            for (bool ok = true; ok;) {
                // the first tile of every CTA is its own index (no atomic on the way
                // to the first load); later ones come from the counter, which
                // hands out the tiles from gridDim.x on
                int next = tile < 0 ? (int)blockIdx.x
                                    : (p.counter ? (int)gridDim.x + atomicAdd(p.counter, 1)
                                                 : tile + (int)gridDim.x);
                if (next >= total_tiles) next = -1;
                const int slot = tpos % S_TILE_SLOTS;
                if (!mbar_wait(&ctl->tile_empty[slot], ((tpos / S_TILE_SLOTS) & 1) ^ 1, &ctl->abort,
                               p.status, p.wait_cycles))
                    break;
                ctl->tile_ring[slot] = next;
                mbar_arrive(&ctl->tile_full[slot]);
                ++tpos;
                if (next < 0) break;
                tile = next;
                const STile tl = s_find_tile(ctl, G, NB, tile);
                const int g0 = ctl->go[tl.g];
                const int nv = min(STOK, ctl->go[tl.g + 1] - g0 - tl.c * STOK);
                const int boxes = (nv + SBOX - 1) / SBOX;
                const int a_row = g0 + tl.c * STOK;
                const int w_row = tl.g * p.N + tl.nt * SWR;
                const uint32_t bytes = C::NW * SMEM_W + boxes * SBOX * SK;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % C::STAGES;
                    if (!mbar_wait(&ctl->empty[s], ((it / C::STAGES) & 1) ^ 1, &ctl->abort, p.status, p.wait_cycles)) {
                        ok = false;
                        break;
                    }
                    if (p.stall) {
                        // test switch: nothing fills this stage, so this wait (and the
                        // MMA issuer's) runs out after the wait limit
                        mbar_wait(&ctl->full[s], (it / C::STAGES) & 1, &ctl->abort, p.status,
                                  p.wait_cycles);
                        ok = false;
                        break;
                    }
                    uint8_t* sW = smem + (size_t)s * C::STAGE;
                    uint8_t* sT = sW + C::NW * SMEM_W;
                    mbar_expect_tx(&ctl->full[s], bytes);
                    tma_load_2d(sW, &tmW0, &ctl->full[s], kb * SK, w_row);
                    if (gate_up) tma_load_2d(sW + SMEM_W, &tmW1, &ctl->full[s], kb * SK, w_row);
                    for (int b = 0; b < boxes; ++b)
                        tma_load_2d(sT + b * SBOX * SK, &tmA, &ctl->full[s], kb * SK, a_row + b * SBOX);
                }
            }
            const uint32_t first = it > (uint32_t)C::STAGES ? it - C::STAGES : 0;
            for (uint32_t j = first; j < it; ++j) mbar_drain(&ctl->full[j % C::STAGES], (j / C::STAGES) & 1);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            uint32_t it = 0, tpos = 0;
            int tile;
            for (bool ok = true; ok;) {
                if (!s_take_tile(ctl, tpos, tile, p.status, p.wait_cycles) || tile < 0) break;
                const STile tl = s_find_tile(ctl, G, NB, tile);
                const int nv = min(STOK, ctl->go[tl.g + 1] - ctl->go[tl.g] - tl.c * STOK);
                const int boxes = (nv + SBOX - 1) / SBOX;
                const uint32_t idesc = idesc_e4m3(SWR, boxes * SBOX);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % C::STAGES;
                    const uint32_t buf = it % S_NBUF;
                    if (!mbar_wait(&ctl->tempty[buf], ((it / S_NBUF) & 1) ^ 1, &ctl->abort, p.status, p.wait_cycles) ||
                        !mbar_wait(&ctl->full[s], (it / C::STAGES) & 1, &ctl->abort, p.status, p.wait_cycles)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t w0 = smem_u32(smem + (size_t)s * C::STAGE);
                    const uint32_t t0 = w0 + C::NW * SMEM_W;
                    const uint32_t d0 = tmem_base + buf * 64;
#pragma unroll
                    for (int k = 0; k < SK / 32; ++k)
                        mma_e4m3(d0, sdesc_sw128(w0 + k * 32), sdesc_sw128(t0 + k * 32), idesc,
                                 k > 0 ? 1u : 0u);
                    if (gate_up) {
#pragma unroll
                        for (int k = 0; k < SK / 32; ++k)
                            mma_e4m3(d0 + STOK, sdesc_sw128(w0 + SMEM_W + k * 32),
                                     sdesc_sw128(t0 + k * 32), idesc, k > 0 ? 1u : 0u);
                    }
                    mma_commit(&ctl->empty[s]);
                    mma_commit(&ctl->tfull[buf]);
                }
            }
            if (it > 0) mbar_drain(&ctl->tfull[(it - 1) % S_NBUF], ((it - 1) / S_NBUF) & 1);
            mbar_drain(&ctl->epi_done, 0, 3 * WAIT_CYCLES);
        }
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(S_TMEM_COLS));
    } else if (warp == 2) {
        // ================= scale loader =================
        uint32_t it = 0, tpos = 0;
        bool ok = true;
        int tile;
        while (ok) {
            if (!s_warp_take_tile(ctl, tpos, tile, p.status, p.wait_cycles)) { ok = false; break; }
            if (tile < 0) break;
            const STile tl = s_find_tile(ctl, G, NB, tile);
            const int g0 = ctl->go[tl.g];
            const int nv = min(STOK, ctl->go[tl.g + 1] - g0 - tl.c * STOK);
            const float* w0 = p.sw0 + ((size_t)tl.g * NB + tl.nt) * KB;
            const float* w1 = gate_up ? p.sw1 + ((size_t)tl.g * NB + tl.nt) * KB : w0;
            const int row = g0 + tl.c * STOK + lane;
            const bool v = lane < nv && row < p.M_total;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int slot = it % S_SCALE_SLOTS;
                bool got = true;
                if (lane == 0)
                    got = mbar_wait(&ctl->sempty[slot], ((it / S_SCALE_SLOTS) & 1) ^ 1, &ctl->abort,
                                    p.status, p.wait_cycles);
                if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) { ok = false; break; }
                SScaleSlot& sl = ctl->scales[slot];
                cp_async4(&sl.sa[lane], v ? p.sa + (size_t)kb * p.M_total + row : p.sa, v ? 4u : 0u);
                if (lane == 0) {
                    cp_async4(&sl.sw[0], w0 + kb, 4u);
                    cp_async4(&sl.sw[1], w1 + kb, 4u);
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
                if (it >= (uint32_t)S_SCALE_LAG) {
                    asm volatile("cp.async.wait_group %0;" ::"n"(S_SCALE_LAG) : "memory");
                    mbar_arrive(&ctl->sfull[(it - S_SCALE_LAG) % S_SCALE_SLOTS]);
                }
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (ok)
            for (uint32_t j = it > (uint32_t)S_SCALE_LAG ? it - S_SCALE_LAG : 0; j < it; ++j)
                mbar_arrive(&ctl->sfull[j % S_SCALE_SLOTS]);
    } else if (warp >= S_EPI0) {
        // ================= epilogue =================
        const int q = warp & 3;                    // TMEM lane quarter
        const int r = q * 32 + lane;               // weight row within the tile
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        uint32_t it = 0, tpos = 0;
        int tcount = 0;
        bool ok = true;
        int tile;
        for (; ok; ++tcount) {
            if (!s_warp_take_tile(ctl, tpos, tile, p.status, p.wait_cycles)) { ok = false; break; }
            if (tile < 0) break;
            const STile tl = s_find_tile(ctl, G, NB, tile);
            const int g0 = ctl->go[tl.g];
            const int nv = min(STOK, ctl->go[tl.g + 1] - g0 - tl.c * STOK);
            const int row0 = g0 + tl.c * STOK;
            float acc0[STOK], acc1[STOK];
#pragma unroll
            for (int i = 0; i < STOK; ++i) acc0[i] = acc1[i] = 0.0f;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int slot = it % S_SCALE_SLOTS;
                const uint32_t buf = it % S_NBUF;
                if (!warp_wait(&ctl->sfull[slot], (it / S_SCALE_SLOTS) & 1, &ctl->abort, p.status, p.wait_cycles) ||
                    !warp_wait(&ctl->tfull[buf], (it / S_NBUF) & 1, &ctl->abort, p.status, p.wait_cycles)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t a[32], b[32];
                const uint32_t taddr = tmem_base + lane_addr + buf * 64;
                tmem_ld32_nowait(taddr, a);
                if (gate_up) tmem_ld32_nowait(taddr + STOK, b);
                tmem_ld_wait(a);
                if (gate_up) reg_after_wait(b);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->tempty[buf]);
                const SScaleSlot& sl = ctl->scales[slot];
                // acc[t] = fma(partial, sa[t] * sw, acc[t]) for the chunk's rows
                // (nv is the same in every thread: at most 8, 16 or 32 columns)
                if (nv <= 8) {
                    fma2_rowcol<8>(acc0, a, sl.sw[0], sl.sa);
                    if (gate_up) fma2_rowcol<8>(acc1, b, sl.sw[1], sl.sa);
                } else if (nv <= 16) {
                    fma2_rowcol<16>(acc0, a, sl.sw[0], sl.sa);
                    if (gate_up) fma2_rowcol<16>(acc1, b, sl.sw[1], sl.sa);
                } else {
                    fma2_rowcol<STOK>(acc0, a, sl.sw[0], sl.sa);
                    if (gate_up) fma2_rowcol<STOK>(acc1, b, sl.sw[1], sl.sa);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->sempty[slot]);
            }
            if (!ok) break;
            if constexpr (gate_up) {
                // h = SiLU(g) * u, SiLU(g) = g / (1 + e^-g); amax of each row over
                // the tile's 128 intermediate indices (the four warps' lanes); only
                // the chunk's nv rows (nv is the same in every thread)
                const int par = tcount & 1;
#pragma unroll
                for (int t = 0; t < STOK; ++t) {
                    if (t >= nv) break;
                    const float gv = acc0[t];
                    const float h = __fdiv_rn(gv, 1.0f + expf(-gv)) * acc1[t];
                    acc0[t] = h;
                    float m = fabsf(h);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                    if (lane == t) ctl->amax[par][q][t] = m;
                }
                __threadfence_block();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->xbar);
                if (!warp_wait(&ctl->xbar, (uint32_t)par, &ctl->abort, p.status, p.wait_cycles)) { ok = false; break; }
                uint8_t* dst = static_cast<uint8_t*>(p.out) + (size_t)row0 * p.N + tl.nt * SWR + r;
#pragma unroll
                for (int t = 0; t < STOK; ++t) {
                    if (t >= nv) break;
                    const float am = fmaxf(fmaxf(ctl->amax[par][0][t], ctl->amax[par][1][t]),
                                           fmaxf(ctl->amax[par][2][t], ctl->amax[par][3][t]));
                    const float scale = tile_scale(am);
                    float qv;
                    if (am == 0.0f) qv = 0.0f;
                    else if (scale >= 0x1p-100f) qv = s_div_rcp(acc0[t], scale, __frcp_rn(scale));
                    else qv = __fdiv_rn(acc0[t], scale);
                    dst[(size_t)t * p.N] = static_cast<uint8_t>(e4m3x2(qv, 0.0f) & 0xFFu);
                    if (r == t) p.out_scales[(size_t)tl.nt * p.M_total + row0 + t] = scale;
                }
            } else if (tl.g >= p.f32_group0) {
                float* dst = p.out2 + (size_t)(row0 - p.f32_row0) * p.N + tl.nt * SWR + r;
#pragma unroll
                for (int t = 0; t < STOK; ++t) {
                    if (t >= nv) break;
                    dst[(size_t)t * p.N] = acc0[t];
                }
            } else {
                uint16_t* dst = static_cast<uint16_t*>(p.out) + (size_t)row0 * p.N + tl.nt * SWR + r;
#pragma unroll
                for (int t = 0; t < STOK; ++t) {
                    if (t >= nv) break;
                    dst[(size_t)t * p.N] = __bfloat16_as_ushort(__float2bfloat16_rn(acc0[t]));
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->epi_done);
    }
}

}  // namespace

int launch_grouped_gemm_small(int mode, const uint8_t* A, const float* sa, int M_total,
                              const int32_t* go, int G, const uint8_t* W0, const uint8_t* W1,
                              const float* sw0, const float* sw1, int N, int Kdim, void* out,
                              float* out_scales, int32_t* status, cudaStream_t st, int f32_group0,
                              int f32_row0, float* out2, int counter_slot, bool counter_zeroed,
                              int max_ctas) {
    if (M_total == 0 || G == 0) return MOE_OK;
    static int sm_count = 0;
    static std::once_flag once;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    std::call_once(once, [&] {
        cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
        cudaFuncSetAttribute(grouped_gemm_small_kernel<0>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)small_smem_bytes<0>());
        cudaFuncSetAttribute(grouped_gemm_small_kernel<1>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)small_smem_bytes<1>());
    });
    if (sm_count <= 0) return cuda_fail(cudaErrorInvalidDevice);
    const bool gu = mode == MOE_GEMM_GATE_UP_SILU_QUANT;
    CUtensorMap mA, mW0, mW1;
    int rc = make_map_2d(&mA, A, (uint64_t)M_total, (uint64_t)Kdim, 1, SBOX, SK);
    if (rc) return rc;
    if ((rc = make_map_2d(&mW0, W0, (uint64_t)G * N, (uint64_t)Kdim, 1, SWR, SK))) return rc;
    if (gu) {
        if ((rc = make_map_2d(&mW1, W1, (uint64_t)G * N, (uint64_t)Kdim, 1, SWR, SK))) return rc;
    } else {
        mW1 = mW0;
    }
    int* counter = status ? status + counter_slot : nullptr;
    if (counter && !counter_zeroed) {
        const cudaError_t ce = cudaMemsetAsync(counter, 0, sizeof(int), st);
        if (ce != cudaSuccess) return cuda_fail(ce);
    }
    if (mode == MOE_GEMM_DOWN_F32) {                // every group's rows in float32
        f32_group0 = 0;
        f32_row0 = 0;
        out2 = static_cast<float*>(out);
    }
    SParams p{M_total, G, N, Kdim, go, sa, sw0, sw1, out, out_scales, status, counter,
              !gu && out2 ? f32_group0 : (1 << 30), f32_row0, out2, pipeline_wait_cycles(),
              pipeline_stall()};
    const long long max_tiles = ((long long)(M_total + STOK - 1) / STOK + G) * (N / SWR);
    const int ctas = max_ctas > 0 && max_ctas < sm_count ? max_ctas : sm_count;
    const int grid = (int)(max_tiles < ctas ? max_tiles : ctas);
    if (gu)
        return launch_pdl(grouped_gemm_small_kernel<1>, dim3(grid), dim3(S_THREADS),
                          small_smem_bytes<1>(), st, mA, mW0, mW1, p);
    return launch_pdl(grouped_gemm_small_kernel<0>, dim3(grid), dim3(S_THREADS),
                      small_smem_bytes<0>(), st, mA, mW0, mW1, p);
}

}  // namespace moe
