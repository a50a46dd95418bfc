// Grouped block-scaled FP8 GEMM for the expert FFNs, on sm_103a tensor cores.
//
// Source: "รายงานเชิงเทคนิคของ DeepSeek-V3" (xyznot.com/th/paper/2412.19437),
// Key ideas, FP8 bullet, and "官方揭秘DeepSeek-V3模型训练全流程"
// (youleyou.com) §4.3: operands are E4M3 with one FP32 scale per 1x128
// activation tile and per 128x128 weight block; the tensor core sums one
// N_c = 128 slab of K, and that partial is promoted to an FP32 accumulator:
//     acc = fma(partial, sa[row, kb] * sw[nb, kb], acc).
// The pages do this on H800 by copying the tensor-core result into CUDA-core
// registers.  Here the slab partial lands in TMEM (two ping-pong buffers);
// epilogue warps read it with tcgen05.ld and promote it in registers while
// the tensor core fills the other buffer.
//
// Kernel shape (one persistent CTA per SM, 384 threads = 3 warpgroups):
//   warp 0      TMA producer: A tile [128 x 128] + B tile [256 x 128] per slab,
//               STAGES-deep shared-memory ring, 128-byte swizzle.
//   warp 1      TMEM allocator and MMA issuer: 4 x tcgen05.mma.kind::f8f6f4
//               (M=128, N=256, K=32) per slab into TMEM buffer (slab & 1).
//   warp 2      scale loader: the 128 activation scales and the two weight
//               scales of each slab go into a shared-memory ring, so the
//               epilogue never waits on global memory.
//   warp 3      idle.  Warpgroup 0 gives its registers away (setmaxnreg 40).
//   warps 4..11 epilogue, two warpgroups with 232 registers per thread; TMEM
//               lane quarter = warp % 4, so thread (warp, lane) owns output
//               row 32 * (warp % 4) + lane of the tile; warpgroup 1 / 2 own
//               half of the 256 columns each.
// Output tile = 128 rows x 256 columns: in GATE_UP mode 128 gate columns and
// the 128 up columns of the same intermediate indices (so SiLU(G) * U and
// the 1x128 re-quantisation of h stay inside one tile), in DOWN mode 256
// consecutive output features.
//
// Tiles are enumerated group-major, then N tile, then M tile: CTAs running
// at the same time share the weight slab of one (group, N tile) and the A
// rows of one group through L2, so each weight byte is read from HBM once.
//
// Every wait is bounded (about 2 s of SM clock); on expiry the kernel records
// MOE_ERR_TIMEOUT in the status word, every role stops, in-flight copies and
// MMAs are waited for (again bounded) and TMEM is released before exit.
#include <cuda.h>
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {
using namespace tc;

constexpr int BM = 128;
constexpr int BK = 128;
constexpr int BN = 256;
constexpr int STAGES = 4;
constexpr int SMEM_A = BM * BK;                 // 16 KB
constexpr int SMEM_B = BN * BK;                 // 32 KB
constexpr int SMEM_STAGE = SMEM_A + SMEM_B;     // 48 KB
constexpr int NUM_EPI_WARPS = 8;
constexpr int EPI_WARP0 = 4;                    // first epilogue warp
constexpr int NUM_THREADS = 128 + 32 * NUM_EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;             // 2 buffers x 256 fp32 columns
constexpr int SCALE_SLOTS = 8;                  // depth of the scale ring
constexpr int SCALE_LAG = 3;                    // copy groups in flight before a slab is published
constexpr int TILE_SLOTS = 4;                   // depth of the tile-index ring
constexpr int TILE_READERS = 2 + NUM_EPI_WARPS; // MMA thread, scale loader, epilogue warps
// Register split: the kernel is compiled for 384 threads x 168 registers
// (64512); warpgroup 0 drops to 40 and the two epilogue warpgroups rise to
// 232: 128 * 40 + 256 * 232 = 64512.  Per SM sub-partition (warps w, w+4,
// w+8): 40 + 232 + 232 = 504 = 3 * 168.  The host refuses to launch unless
// the compiled register count is exactly LAUNCH_REGS.
constexpr int LAUNCH_REGS = 168;
constexpr int CTRL_REGS = 40;
constexpr int EPI_REGS = 232;
static_assert(128 * CTRL_REGS + 256 * EPI_REGS <= NUM_THREADS * LAUNCH_REGS, "register split");

struct alignas(16) ScaleSlot {
    float sa[BM];                               // activation scale of each tile row
    float sw[4];                                // weight scale of column half 0 and 1
};

struct alignas(16) Ctl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t xbar;                              // amax exchange between the epilogue warpgroups
    uint64_t epi_done;                          // every epilogue warp finished with TMEM
    uint64_t sfull[SCALE_SLOTS];
    uint64_t sempty[SCALE_SLOTS];
    uint64_t tile_full[TILE_SLOTS];
    uint64_t tile_empty[TILE_SLOTS];
    int tile_ring[TILE_SLOTS];                  // tile indices in processing order; -1 ends
    uint32_t tmem_base;
    int abort;
    int total_tiles;
    int pad;
    float amax_x[2][2][BM];                     // [tile parity][warpgroup][row]
    float amax_y[2][2][BM];                     // second block of a row (gate/up gradient mode)
    ScaleSlot scales[SCALE_SLOTS];
    int go[kMaxGroups + 1];                     // group row offsets
    int tile_start[kMaxGroups + 1];             // first tile of each group
};

constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * SMEM_STAGE + sizeof(Ctl);

struct Params {
    int mode;
    int M_total;
    int G;
    int N;
    int Kdim;
    const int32_t* go;
    const float* sa;
    const float* sw0;
    const float* sw1;
    void* out;
    float* out_scales;
    int32_t* status;
    int* counter;                               // next unclaimed tile (nullable: static order)
    const uint16_t* dH;                         // gradient of h [M_total, N] bf16 (gradient mode)
    // DOWN: rows of groups >= f32_group0 go to out2 (float32, row - f32_row0);
    // the others to out (bf16)
    int f32_group0;
    int f32_row0;
    float* out2;
    long long wait_cycles;                      // limit of every pipeline wait (SM clock cycles)
    int stall;                                  // test switch: the producer issues no loads
};

// ----------------------------------------------------------- tile lookup
struct Tile {
    int g, nt, mt;
};

__device__ __forceinline__ Tile find_tile(const Ctl* ctl, int G, int tile) {
    int lo = 0, hi = G;                     // tile_start[lo] <= tile < tile_start[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (ctl->tile_start[mid] <= tile) lo = mid; else hi = mid;
    }
    const int m = max(0, ctl->go[lo + 1] - ctl->go[lo]);
    const int mtiles = (m + BM - 1) / BM;
    const int local = tile - ctl->tile_start[lo];
    return Tile{lo, local / mtiles, local % mtiles};
}

// x / scale correctly rounded (the IEEE quotient) without a division
// instruction, from r = RN(1 / scale): y = RN(x r) is within 2 ulps of the
// quotient; one correction step q1 = RN(y + RN(x - scale y) r) makes it
// faithful, and a second step from a faithful quotient with the correctly
// rounded reciprocal rounds correctly (Markstein, IBM J. Res. Dev. 34(1),
// 1990; the residual x - scale q1 is exact in one FMA).  The correction sums
// turn a -0 quotient into +0, so the sign is taken from x (scale > 0).  The
// scale must be far from underflow.
__device__ __forceinline__ float div_rcp(float x, float scale, float r) {
    const float y = x * r;
    const float q1 = fmaf(fmaf(-scale, y, x), r, y);
    return copysignf(fmaf(fmaf(-scale, q1, x), r, q1), x);
}
__device__ __forceinline__ uint32_t quant4_rcp(float a, float b, float c, float d, float scale,
                                               float r) {
    const uint32_t lo = e4m3x2(div_rcp(a, scale, r), div_rcp(b, scale, r));
    const uint32_t hi = e4m3x2(div_rcp(c, scale, r), div_rcp(d, scale, r));
    return lo | (hi << 16);
}

// 8 x 8 transpose of 16-byte chunks within each octet of lanes (lanes 8q ..
// 8q + 7).  Before: lane j of the octet holds chunks 0..7 of its own output
// row in x[0..7].  After: x[c] holds chunk j of the row of octet lane c.
// Three butterfly stages (lane distance 4, 2, 1), each swapping the
// off-diagonal sub-blocks of the blocks left by the stage before, so that a
// store instruction afterwards writes 128 contiguous bytes of four rows
// instead of 16 bytes of 32 rows.
__device__ __forceinline__ void octet_transpose(uint32_t (&x)[8][4]) {
    const int j = threadIdx.x & 7;
#pragma unroll
    for (int k = 4; k > 0; k >>= 1) {
        const bool upper = (j & k) != 0;
#pragma unroll
        for (int c0 = 0; c0 < 8; ++c0) {
            if (c0 & k) continue;
            const int c1 = c0 | k;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t send = upper ? x[c0][w] : x[c1][w];
                const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, k);
                if (upper) x[c0][w] = recv; else x[c1][w] = recv;
            }
        }
    }
}
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// The next tile index from the ring (-1: no more tiles); false when the wait
// gave up.  Single-thread form (MMA issuer) and warp form.
__device__ __forceinline__ bool take_tile(Ctl* ctl, uint32_t& tpos, int& tile, int32_t* status, long long limit) {
    const int slot = tpos % TILE_SLOTS;
    if (!mbar_wait(&ctl->tile_full[slot], (tpos / TILE_SLOTS) & 1, &ctl->abort, status, limit)) return false;
    tile = ctl->tile_ring[slot];
    mbar_arrive(&ctl->tile_empty[slot]);
    ++tpos;
    return true;
}
__device__ __forceinline__ bool warp_take_tile(Ctl* ctl, uint32_t& tpos, int& tile, int32_t* status, long long limit) {
    const int slot = tpos % TILE_SLOTS;
    if (!warp_wait(&ctl->tile_full[slot], (tpos / TILE_SLOTS) & 1, &ctl->abort, status, limit)) return false;
    tile = ctl->tile_ring[slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&ctl->tile_empty[slot]);
    ++tpos;
    return true;
}

// ---------------------------------------------------------------- kernel
// MODE 0: down projection; 1: gate/up + SiLU + re-quantisation; 2: gate/up
// recomputed for the input gradient (SiLU backward against dH, [dG | dU]
// re-quantised).
template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB0,
                            const __grid_constant__ CUtensorMap tmB1, const Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    Ctl* ctl = reinterpret_cast<Ctl*>(smem + (size_t)STAGES * SMEM_STAGE);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr bool gate_up = MODE != 0;
    constexpr bool dgrad = MODE == 2;
    const int NT = gate_up ? p.N / 128 : (p.N + BN - 1) / BN;
    const int NB = p.N / 128;
    const int KB = p.Kdim / BK;
    const int G = p.G;

    // ---- prologue.  Barriers, TMEM and the tensor-map prefetch touch only this
    // CTA's own memory, so they are set up before waiting for the kernel this
    // launch depends on (programmatic dependent launch); the group offsets are
    // that kernel's output.
    if (warp == 0) {
        if (lane == 0) {
            for (int s = 0; s < STAGES; ++s) {
                mbar_init(&ctl->full[s], 1);
                mbar_init(&ctl->empty[s], 1);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(&ctl->tfull[b], 1);
                mbar_init(&ctl->tempty[b], NUM_EPI_WARPS);
            }
            for (int s = 0; s < SCALE_SLOTS; ++s) {
                mbar_init(&ctl->sfull[s], 32);   // one arrival per loader lane
                mbar_init(&ctl->sempty[s], NUM_EPI_WARPS);
            }
            for (int s = 0; s < TILE_SLOTS; ++s) {
                mbar_init(&ctl->tile_full[s], 1);
                mbar_init(&ctl->tile_empty[s], TILE_READERS);
            }
            mbar_init(&ctl->xbar, NUM_EPI_WARPS);
            mbar_init(&ctl->epi_done, NUM_EPI_WARPS);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB0);
            if (gate_up) tma_prefetch_desc(&tmB1);
        }
    } else if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&ctl->tmem_base)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    griddep_wait();
    griddep_launch();
    // every thread copies a share of the group offsets (one round of loads
    // instead of one per 32 groups), then warp 0 scans them:
    // tile_start[g] = sum_{g' < g} ceil(m_g' / 128) * NT
    for (int g = threadIdx.x; g <= G; g += NUM_THREADS) ctl->go[g] = p.go[g];
    __syncthreads();
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base <= G; base += 32) {
            const int g = base + lane;
            int v = 0;
            if (g < G) {
                const int m = max(0, ctl->go[g + 1] - ctl->go[g]);
                v = (m + BM - 1) / BM * NT;
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

    // Each warpgroup's role code sits under its own setmaxnreg, so the
    // register allocator sees the budget of the region it is compiling.
    if (warp < EPI_WARP0) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(CTRL_REGS));
      // (role code of warpgroup 0 below is indented one level less than its scope)
      if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            uint32_t it = 0, tpos = 0;
            bool ok = true;
            int tile = -1;
            while (ok) {
                // claim the next tile (adjacent claims share a weight panel, so
                // CTAs that claim them together stream it from HBM once) and
                // publish it to the other roles
                // the first tile of every CTA is its own index (no atomic on the way
                // to the first load); later ones come from the counter, which
                // hands out the tiles from gridDim.x on
                int next = tile < 0 ? (int)blockIdx.x
                                    : (p.counter ? (int)gridDim.x + atomicAdd(p.counter, 1)
                                                 : tile + (int)gridDim.x);
                if (next >= total_tiles) next = -1;
                const int slot = tpos % TILE_SLOTS;
                if (!mbar_wait(&ctl->tile_empty[slot], ((tpos / TILE_SLOTS) & 1) ^ 1, &ctl->abort,
                               p.status, p.wait_cycles)) {
                    ok = false;
                    break;
                }
                ctl->tile_ring[slot] = next;
                mbar_arrive(&ctl->tile_full[slot]);
                ++tpos;
                if (next < 0) break;
                tile = next;
                const Tile tl = find_tile(ctl, G, tile);
                const int a_row = ctl->go[tl.g] + tl.mt * BM;
                int b0_row, b1_row;
                bool has_b1;
                if (gate_up) {
                    b0_row = tl.g * p.N + tl.nt * 128;
                    b1_row = b0_row;
                    has_b1 = true;
                } else {
                    b0_row = tl.g * p.N + tl.nt * BN;
                    b1_row = b0_row + 128;
                    has_b1 = tl.nt * BN + 128 < p.N;
                }
                const uint32_t bytes = SMEM_A + 128 * BK * (has_b1 ? 2 : 1);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait(&ctl->empty[s], ph ^ 1, &ctl->abort, p.status, p.wait_cycles)) { ok = false; break; }
                    if (p.stall) {
                        // test switch: nothing fills this stage, so this wait (and the
                        // MMA issuer's) runs out after the wait limit
                        mbar_wait(&ctl->full[s], ph, &ctl->abort, p.status, p.wait_cycles);
                        ok = false;
                        break;
                    }
                    uint8_t* sA = smem + (size_t)s * SMEM_STAGE;
                    uint8_t* sB = sA + SMEM_A;
                    mbar_expect_tx(&ctl->full[s], bytes);
                    tma_load_2d(sA, &tmA, &ctl->full[s], kb * BK, a_row);
                    tma_load_2d(sB, &tmB0, &ctl->full[s], kb * BK, b0_row);
                    if (has_b1)
                        tma_load_2d(sB + 128 * BK, gate_up ? &tmB1 : &tmB0, &ctl->full[s],
                                    kb * BK, b1_row);
                }
            }
            // make sure no copy is still landing in shared memory when the CTA exits
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
                if (!take_tile(ctl, tpos, tile, p.status, p.wait_cycles)) break;
                if (tile < 0) break;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    const uint32_t buf = it & 1;
                    const uint32_t tph = (it >> 1) & 1;
                    if (!mbar_wait(&ctl->tempty[buf], tph ^ 1, &ctl->abort, p.status, p.wait_cycles)) { ok = false; break; }
                    if (!mbar_wait(&ctl->full[s], ph, &ctl->abort, p.status, p.wait_cycles)) { ok = false; break; }
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
            // wait for the last MMAs, and for every epilogue warp to finish
            // reading TMEM, before TMEM is released (both bounded)
            if (it > 0) mbar_drain(&ctl->tfull[(it - 1) & 1], ((it - 1) >> 1) & 1);
            // (longer than any single wait, so an aborting epilogue is out first)
            mbar_drain(&ctl->epi_done, 0, 3 * WAIT_CYCLES);
        }
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(TMEM_COLS));
    } else if (warp == 2) {
        // ================= scale loader =================
        // Slot j of the ring holds slab j's 128 activation scales (row order of
        // the tile, 0 for rows outside the group) and the weight scale of each
        // 128-column half of the output tile.
        uint32_t it = 0, tpos = 0;
        bool ok = true;
        int tile;
        while (ok) {
            if (!warp_take_tile(ctl, tpos, tile, p.status, p.wait_cycles)) { ok = false; break; }
            if (tile < 0) break;
            const Tile tl = find_tile(ctl, G, tile);
            const int g0 = ctl->go[tl.g];
            const int m_g = max(0, ctl->go[tl.g + 1] - g0);
            const float* w0;
            const float* w1;
            if (gate_up) {
                w0 = p.sw0 + ((size_t)tl.g * NB + tl.nt) * KB;
                w1 = p.sw1 + ((size_t)tl.g * NB + tl.nt) * KB;
            } else {
                w0 = p.sw0 + ((size_t)tl.g * NB + tl.nt * 2) * KB;
                w1 = (tl.nt * 2 + 1 < NB) ? w0 + KB : w0;
            }
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int slot = it % SCALE_SLOTS;
                const uint32_t ph = (it / SCALE_SLOTS) & 1;
                bool got = true;
                if (lane == 0) {
                    // The loader usually runs ahead with the ring full.  It shares its
                    // SM sub-partition with two epilogue warps, so it sleeps between
                    // polls (at most 64 x 128 ns) before the bounded wait.
                    for (int spin = 0; spin < 64 && !mbar_test(&ctl->sempty[slot], ph ^ 1); ++spin)
                        __nanosleep(128);
                    got = mbar_wait(&ctl->sempty[slot], ph ^ 1, &ctl->abort, p.status, p.wait_cycles);
                }
                if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) { ok = false; break; }
                // 4-byte asynchronous copies; rows outside the group are zero-filled
                // (source size 0).  One commit group per slab; slab it - SCALE_LAG is
                // announced on its sfull barrier once its group has landed, so the
                // loader runs up to SCALE_SLOTS slabs ahead and each slab is published
                // as soon as its own copies are complete.  (An mbarrier arrive tied
                // to cp.async completion would wait for every earlier copy of the
                // thread, including the newer slabs' copies in flight.)
                ScaleSlot& sl = ctl->scales[slot];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = lane * 4 + j;
                    const int lrow = tl.mt * BM + r;
                    const int grow = g0 + lrow;
                    const bool v = lrow < m_g && grow < p.M_total;
                    const float* src = v ? p.sa + (size_t)kb * p.M_total + grow : p.sa;
                    cp_async4(&sl.sa[r], src, v ? 4u : 0u);
                }
                if (lane == 0) {
                    cp_async4(&sl.sw[0], w0 + kb, 4u);
                    cp_async4(&sl.sw[1], w1 + kb, 4u);
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
                if (it >= (uint32_t)SCALE_LAG) {
                    asm volatile("cp.async.wait_group %0;" ::"n"(SCALE_LAG) : "memory");
                    mbar_arrive(&ctl->sfull[(it - SCALE_LAG) % SCALE_SLOTS]);
                }
            }
        }
        // publish the slabs still in flight (on abort nobody waits for them)
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
        uint32_t it = 0, tpos = 0;
        int tcount = 0;
        bool ok = true;
        int tile;
        for (; ok; ++tcount) {
            if (!warp_take_tile(ctl, tpos, tile, p.status, p.wait_cycles)) { ok = false; break; }
            if (tile < 0) break;
            const Tile tl = find_tile(ctl, G, tile);
            const int g0 = ctl->go[tl.g];
            const int m_g = max(0, ctl->go[tl.g + 1] - g0);
            const int lrow = tl.mt * BM + row;
            const int grow = g0 + lrow;
            const bool valid = lrow < m_g && grow < p.M_total;
            const bool cols_valid = gate_up || tl.nt * 2 + wg < NB;
            // TMEM columns of this thread's two 64-column chunks.  GATE_UP: gate
            // cols wg*64 + [0,64) then up cols 128 + wg*64 + [0,64); DOWN: cols
            // wg*128 + [0,128).
            const uint32_t c0 = gate_up ? wg * 64 : wg * 128;
            const uint32_t c1 = gate_up ? 128 + wg * 64 : wg * 128 + 64;
            float acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
            // Software pipeline over the four 32-column chunks of a slab: the load
            // of chunk j+1 is in flight while chunk j is promoted, the TMEM buffer
            // is released as soon as its last chunk is in registers, and the next
            // slab's first chunk loads while this slab's last chunk is promoted.
            uint32_t a[32], b[32];
            float s_lo = 0.0f, s_hi = 0.0f;
            // scales of slab `it` from the ring; false when the wait gave up
            auto take_scales = [&](uint32_t i, float& lo, float& hi) -> bool {
                const int slot = i % SCALE_SLOTS;
                if (!warp_wait(&ctl->sfull[slot], (i / SCALE_SLOTS) & 1, &ctl->abort, p.status, p.wait_cycles)) return false;
                const ScaleSlot& sl = ctl->scales[slot];
                const float sa = sl.sa[row];
                lo = sa * (gate_up ? sl.sw[0] : sl.sw[wg]);
                hi = sa * (gate_up ? sl.sw[1] : sl.sw[wg]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->sempty[slot]);
                return true;
            };
            // A warp whose 32 rows all lie past the group's last row (the padding
            // of a group's last tile) keeps the barrier protocol but neither
            // reads TMEM nor promotes.
            const bool warp_active = tl.mt * BM + quarter * 32 < m_g;
            if (!warp_active) {
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    float lo, hi;
                    if (!take_scales(it, lo, hi) ||
                        !warp_wait(&ctl->tfull[it & 1], (it >> 1) & 1, &ctl->abort, p.status, p.wait_cycles)) {
                        ok = false;
                        break;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctl->tempty[it & 1]);
                }
            } else if (KB > 0) {
                if (!take_scales(it, s_lo, s_hi) ||
                    !warp_wait(&ctl->tfull[it & 1], (it >> 1) & 1, &ctl->abort, p.status, p.wait_cycles)) {
                    ok = false;
                } else {
                    tc_fence_after();
                    tmem_ld32_nowait(tmem_base + lane_addr + (it & 1) * BN + c0, a);
                    tmem_ld_wait(a);
                }
            }
            for (int kb = 0; ok && warp_active && kb < KB; ++kb, ++it) {
                const uint32_t tbase = tmem_base + lane_addr + (it & 1) * BN;
                tmem_ld32_nowait(tbase + c0 + 32, b);
                fma2_scale<32>(acc, a, s_lo);
                tmem_ld_wait(b);
                tmem_ld32_nowait(tbase + c1, a);
                fma2_scale<32>(acc + 32, b, s_lo);
                tmem_ld_wait(a);
                tmem_ld32_nowait(tbase + c1 + 32, b);
                fma2_scale<32>(acc + 64, a, s_hi);
                tmem_ld_wait(b);
                // the whole slab is in registers: hand the TMEM buffer back
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->tempty[it & 1]);
                const float last_hi = s_hi;
                if (kb + 1 < KB) {
                    if (!take_scales(it + 1, s_lo, s_hi) ||
                        !warp_wait(&ctl->tfull[(it + 1) & 1], ((it + 1) >> 1) & 1, &ctl->abort, p.status, p.wait_cycles)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    tmem_ld32_nowait(tmem_base + lane_addr + ((it + 1) & 1) * BN + c0, a);
                }
                fma2_scale<32>(acc + 96, b, last_hi);
                if (kb + 1 < KB) tmem_ld_wait(a);
            }
            if (!ok) break;
            // ---- tile finalisation
            if constexpr (gate_up) {
                float amax = 0.0f, amax2 = 0.0f;
                if (warp_active) {
                    if constexpr (!dgrad) {
                        // h = SiLU(g) * u with SiLU(g) = g / (1 + e^-g)
#pragma unroll
                        for (int i = 0; i < 64; ++i) {
                            const float gv = acc[i];
                            const float h = __fdiv_rn(gv, 1.0f + expf(-gv)) * acc[64 + i];
                            acc[i] = h;
                            amax = fmaxf(amax, fabsf(h));
                        }
                    } else {
                        // sigma = 1 / (1 + e^-g); dG = dH u sigma (1 + g (1 - sigma)),
                        // dU = dH g sigma; acc[0, 64) becomes dG, acc[64, 128) dU
                        const uint16_t* dhr = p.dH + (size_t)(valid ? grow : 0) * p.N + tl.nt * 128 + wg * 64;
#pragma unroll
                        for (int j = 0; j < 64; j += 8) {
                            const uint4 v = valid ? *reinterpret_cast<const uint4*>(dhr + j)
                                                  : make_uint4(0u, 0u, 0u, 0u);
                            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float dh = bf16_bits_to_float(static_cast<uint16_t>(
                                    (q & 1) ? (w4[q >> 1] >> 16) : (w4[q >> 1] & 0xFFFFu)));
                                const float gv = acc[j + q], uv = acc[64 + j + q];
                                const float sg = __fdiv_rn(1.0f, 1.0f + expf(-gv));
                                const float dG = dh * uv * sg * (1.0f + gv * (1.0f - sg));
                                const float dU = dh * gv * sg;
                                acc[j + q] = dG;
                                acc[64 + j + q] = dU;
                                amax = fmaxf(amax, fabsf(dG));
                                amax2 = fmaxf(amax2, fabsf(dU));
                            }
                        }
                    }
                }
                // Exchange the row's amax with the other warpgroup.  One xbar phase per
                // tile: no warp can arrive for tile n+1 before all arrived for tile n,
                // and the double-buffered slots keep tile n's values until then.
                const int par = tcount & 1;
                ctl->amax_x[par][wg][row] = amax;
                if constexpr (dgrad) ctl->amax_y[par][wg][row] = amax2;
                __threadfence_block();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->xbar);
                if (!warp_wait(&ctl->xbar, (uint32_t)par, &ctl->abort, p.status, p.wait_cycles)) { ok = false; break; }
                amax = fmaxf(ctl->amax_x[par][0][row], ctl->amax_x[par][1][row]);
                if constexpr (dgrad) amax2 = fmaxf(ctl->amax_y[par][0][row], ctl->amax_y[par][1][row]);
                // GATE_UP: one 1x128 block of h (columns 128 nt ..); gradient mode: the
                // block of dG (columns 128 nt .. of [dG | dU]) and that of dU (N + 128 nt ..)
                const int out_ld = dgrad ? 2 * p.N : p.N;
#pragma unroll
                for (int half = 0; half < (dgrad ? 2 : 1); ++half) {
                    const float am = half ? amax2 : amax;
                    const float scale = tile_scale(am);
                    // a tile scale below 2^-100 (amax below ~2^-91) takes IEEE division
                    const bool fast_div = scale >= 0x1p-100f;
                    const float rs = __frcp_rn(scale);
                    if (valid) {
                        uint8_t* dst = static_cast<uint8_t*>(p.out) + (size_t)grow * out_ld + half * p.N +
                                       tl.nt * 128 + wg * 64;
#pragma unroll
                        for (int j = 0; j < 64; j += 16) {
                            const float* v = acc + half * 64 + j;
                            uint4 o;
                            if (am == 0.0f) {
                                o = make_uint4(0u, 0u, 0u, 0u);
                            } else if (!fast_div) {
                                o.x = quant4(v[0], v[1], v[2], v[3], scale);
                                o.y = quant4(v[4], v[5], v[6], v[7], scale);
                                o.z = quant4(v[8], v[9], v[10], v[11], scale);
                                o.w = quant4(v[12], v[13], v[14], v[15], scale);
                            } else {
                                o.x = quant4_rcp(v[0], v[1], v[2], v[3], scale, rs);
                                o.y = quant4_rcp(v[4], v[5], v[6], v[7], scale, rs);
                                o.z = quant4_rcp(v[8], v[9], v[10], v[11], scale, rs);
                                o.w = quant4_rcp(v[12], v[13], v[14], v[15], scale, rs);
                            }
                            *reinterpret_cast<uint4*>(dst + j) = o;
                        }
                        if (wg == 0)
                            p.out_scales[(size_t)(half * NB + tl.nt) * p.M_total + grow] = scale;
                    }
                }
            } else if (warp_active && cols_valid) {
                // Down projection: this thread holds 128 consecutive output columns of
                // its row.  The lanes of each octet trade 16-byte chunks (octet_transpose)
                // so that every store writes 128 contiguous bytes of one row per octet.
                // Octet lane c's row is this warp's row 8 (lane / 8) + c.
                const int j = lane & 7;
                const int orow0 = (lane & ~7);              // lane of octet row 0
                const int col0 = tl.nt * BN + wg * 128;
                uint32_t vmask = 0;                         // bit c: octet row c is an output row
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int lr = tl.mt * BM + quarter * 32 + orow0 + c;
                    if (lr < m_g && g0 + lr < p.M_total) vmask |= 1u << c;
                }
                const int grow0 = g0 + tl.mt * BM + quarter * 32 + orow0;
                uint32_t x[8][4];
                if (tl.g >= p.f32_group0) {
                    // float32 rows: 32 chunks of four values, in four octet blocks
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
#pragma unroll
                        for (int c = 0; c < 8; ++c)
#pragma unroll
                            for (int w = 0; w < 4; ++w) x[c][w] = __float_as_uint(acc[b * 32 + c * 4 + w]);
                        octet_transpose(x);
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            if (vmask >> c & 1u) {
                                float* dst = p.out2 + (size_t)(grow0 + c - p.f32_row0) * p.N + col0 + b * 32 + j * 4;
                                *reinterpret_cast<uint4*>(dst) = make_uint4(x[c][0], x[c][1], x[c][2], x[c][3]);
                            }
                    }
                } else {
                    // bf16 rows: 16 chunks of eight values, in two octet blocks
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
#pragma unroll
                        for (int c = 0; c < 8; ++c)
#pragma unroll
                            for (int w = 0; w < 4; ++w)
                                x[c][w] = bf16x2_bits(acc[b * 64 + c * 8 + 2 * w], acc[b * 64 + c * 8 + 2 * w + 1]);
                        octet_transpose(x);
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            if (vmask >> c & 1u) {
                                uint16_t* dst = static_cast<uint16_t*>(p.out) + (size_t)(grow0 + c) * p.N + col0 +
                                                b * 64 + j * 8;
                                *reinterpret_cast<uint4*>(dst) = make_uint4(x[c][0], x[c][1], x[c][2], x[c][3]);
                            }
                    }
                }
            }
        }
        // this warp's TMEM reads are complete: warp 1 may release TMEM
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->epi_done);
    }
    // No code after the role branches: each role runs under its own register budget.
}

// ------------------------------------------------------------ host side
}  // namespace

int launch_grouped_gemm(int mode, const uint8_t* A, const float* sa, int M_total,
                        const int32_t* go, int G, const uint8_t* W0, const uint8_t* W1,
                        const float* sw0, const float* sw1, int N, int Kdim, void* out,
                        float* out_scales, int32_t* status, cudaStream_t st, const uint16_t* dH,
                        int f32_group0, int f32_row0, float* out2, int counter_slot,
                        bool counter_zeroed, int max_ctas) {
    if (M_total == 0 || G == 0) return MOE_OK;
    static int sm_count = 0;
    static std::once_flag once;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    static int num_regs[3] = {0, 0, 0};
    std::call_once(once, [&] {
        cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
        cudaFuncSetAttribute(grouped_gemm_fp8_kernel<0>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        cudaFuncSetAttribute(grouped_gemm_fp8_kernel<1>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        cudaFuncSetAttribute(grouped_gemm_fp8_kernel<2>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, grouped_gemm_fp8_kernel<0>) == cudaSuccess)
            num_regs[0] = fa.numRegs;
        if (cudaFuncGetAttributes(&fa, grouped_gemm_fp8_kernel<1>) == cudaSuccess)
            num_regs[1] = fa.numRegs;
        if (cudaFuncGetAttributes(&fa, grouped_gemm_fp8_kernel<2>) == cudaSuccess)
            num_regs[2] = fa.numRegs;
    });
    if (sm_count <= 0) return cuda_fail(cudaErrorInvalidDevice);
    // The warpgroups re-split the registers the CTA is launched with; launching
    // with fewer than LAUNCH_REGS per thread would leave setmaxnreg.inc waiting.
    const bool down = mode == MOE_GEMM_DOWN || mode == MOE_GEMM_DOWN_F32;
    const int kmode = down ? 0 : (mode == MOE_GEMM_GATE_UP_SILU_QUANT ? 1 : 2);
    const bool gu = kmode != 0;
    if (num_regs[kmode] != LAUNCH_REGS) return cuda_fail(cudaErrorInvalidConfiguration);
    CUtensorMap mA, mB0, mB1;
    int rc = make_map_2d(&mA, A, (uint64_t)M_total, (uint64_t)Kdim, 1, 128, 128);
    if (rc) return rc;
    rc = make_map_2d(&mB0, W0, (uint64_t)G * N, (uint64_t)Kdim, 1, 128, 128);
    if (rc) return rc;
    if (gu) {
        rc = make_map_2d(&mB1, W1, (uint64_t)G * N, (uint64_t)Kdim, 1, 128, 128);
        if (rc) return rc;
    } else {
        mB1 = mB0;
    }
    // status[counter_slot] is this call's tile counter (dynamic schedule; zeroed
    // here unless the caller already did); without a status buffer the tiles
    // are taken in a fixed order
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
    Params p{mode, M_total, G, N, Kdim, go, sa, sw0, sw1, out, out_scales, status, counter, dH,
             down && out2 ? f32_group0 : (1 << 30), f32_row0, out2, pipeline_wait_cycles(),
             pipeline_stall()};
    const int NT = gu ? N / 128 : (N + BN - 1) / BN;
    const long long max_tiles = ((long long)(M_total + BM - 1) / BM + G) * NT;
    const int ctas = max_ctas > 0 && max_ctas < sm_count ? max_ctas : sm_count;
    const int grid = (int)(max_tiles < ctas ? max_tiles : ctas);
    auto kernel = kmode == 1 ? grouped_gemm_fp8_kernel<1>
                  : kmode == 2 ? grouped_gemm_fp8_kernel<2> : grouped_gemm_fp8_kernel<0>;
    return launch_pdl(kernel, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, st, mA, mB0, mB1, p);
}

}  // namespace moe
