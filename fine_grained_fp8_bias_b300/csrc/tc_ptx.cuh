// tcgen05 / TMA / mbarrier building blocks shared by the tensor-core kernels
// of libmoefp8 (grouped FP8 GEMM and router logits), written as inline PTX
// for sm_103a.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {
namespace tc {

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded waits: by default about 2 s of SM clock (the GEMMs take the limit
// of their pipeline waits from the launch, see moe_set_pipeline_wait_limit).
// The clock is read only every 64 polls, so an unsatisfied wait costs little
// more than the poll itself.  On expiry the waiter records MOE_ERR_TIMEOUT,
// raises the CTA's abort flag (which every other wait checks) and returns
// false.
constexpr long long WAIT_CYCLES = 4000000000LL;

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* abort,
                                          int32_t* status, long long limit = WAIT_CYCLES) {
    if (mbar_test(bar, parity)) return true;
    const long long t0 = clock64();
    const uint32_t every = limit < 1000000 ? 0u : 63u;   // short limits: read the clock each poll
    for (uint32_t i = 1;; ++i) {
        if (mbar_test(bar, parity)) return true;
        if ((i & every) == 0) {
            if (*reinterpret_cast<volatile int*>(abort)) return false;
            if (clock64() - t0 > limit) {
                atomicExch(abort, 1);
                flag_status(status, MOE_ERR_TIMEOUT);
                return false;
            }
        }
    }
}
// Warp-uniform bounded wait: every lane observes the completed phase before
// any lane goes on (the epilogue's tcgen05.ld is .sync.aligned), and all
// lanes agree on giving up.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* abort,
                                          int32_t* status, long long limit = WAIT_CYCLES) {
    const int lane = threadIdx.x & 31;
    const long long t0 = clock64();
    const uint32_t every = limit < 1000000 ? 0u : 63u;
    for (uint32_t i = 0;; ++i) {
        const bool ready = mbar_test(bar, parity);
        if (__all_sync(0xffffffffu, ready)) return true;
        if ((i & every) == every) {
            int stop = 0;
            if (lane == 0) {
                if (*reinterpret_cast<volatile int*>(abort)) {
                    stop = 1;
                } else if (clock64() - t0 > limit) {
                    atomicExch(abort, 1);
                    flag_status(status, MOE_ERR_TIMEOUT);
                    stop = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) return false;
        }
    }
}
// Wait used on the way out: only bounded by time, ignores the abort flag.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity,
                                           long long limit = WAIT_CYCLES) {
    const long long t0 = clock64();
    while (!mbar_test(bar, parity))
        if (clock64() - t0 > limit) return;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}
// 4-byte global -> shared copy; src_bytes = 0 writes zero without reading.
__device__ __forceinline__ void cp_async4(void* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with 128-byte swizzle: rows of 128 bytes, 8-row swizzle atoms of 1024
// bytes stacked along M/N (stride byte offset 1024), descriptor version 1,
// layout type 2 = 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma.kind::f8f6f4: D float32 (bits 4-5 =
// 1), A and B E4M3 (format 0), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// Instruction descriptor of tcgen05.mma.kind::f16 with bf16 A and B (format
// 1 at bits 7-9 and 10-12), float32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 consecutive fp32 TMEM columns of this thread's lane (no wait).
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// acc[2i..2i+1] = fma(v[2i..2i+1], s, acc[..]) with the packed two-lane
// float32 FMA of sm_100+ (two independent round-to-nearest FMAs: the same
// bits as two fmaf calls, half the instructions).
template <int N>
__device__ __forceinline__ void fma2_scale(float* acc, const uint32_t* v, float s) {
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        asm("{\n\t.reg .b64 d, a, b;\n\t"
            "mov.b64 d, {%0, %1};\n\t"
            "mov.b64 a, {%2, %3};\n\t"
            "mov.b64 b, {%4, %4};\n\t"
            "fma.rn.f32x2 d, a, b, d;\n\t"
            "mov.b64 {%0, %1}, d;\n\t}"
            : "+f"(acc[i]), "+f"(acc[i + 1])
            : "r"(v[i]), "r"(v[i + 1]), "f"(s));
    }
}

// acc[i] = fma(v[i], sa * sb[i], acc[i]) for N columns, sa * sb[i] a float32
// product (packed two-lane multiply and FMA, the same bits as mulf / fmaf);
// sb points to 16-byte aligned shared memory.
template <int N>
__device__ __forceinline__ void fma2_rowcol(float* acc, const uint32_t* v, float sa, const float* sb) {
#pragma unroll
    for (int i = 0; i < N; i += 4) {
        const float4 s4 = *reinterpret_cast<const float4*>(sb + i);
        asm("{\n\t.reg .b64 d, a, s, t;\n\t"
            "mov.b64 d, {%0, %1};\n\t"
            "mov.b64 a, {%2, %3};\n\t"
            "mov.b64 s, {%4, %5};\n\t"
            "mov.b64 t, {%6, %6};\n\t"
            "mul.rn.f32x2 s, s, t;\n\t"
            "fma.rn.f32x2 d, a, s, d;\n\t"
            "mov.b64 {%0, %1}, d;\n\t}"
            : "+f"(acc[i]), "+f"(acc[i + 1])
            : "r"(v[i]), "r"(v[i + 1]), "f"(s4.x), "f"(s4.y), "f"(sa));
        asm("{\n\t.reg .b64 d, a, s, t;\n\t"
            "mov.b64 d, {%0, %1};\n\t"
            "mov.b64 a, {%2, %3};\n\t"
            "mov.b64 s, {%4, %5};\n\t"
            "mov.b64 t, {%6, %6};\n\t"
            "mul.rn.f32x2 s, s, t;\n\t"
            "fma.rn.f32x2 d, a, s, d;\n\t"
            "mov.b64 {%0, %1}, d;\n\t}"
            : "+f"(acc[i + 2]), "+f"(acc[i + 3])
            : "r"(v[i + 2]), "r"(v[i + 3]), "f"(s4.z), "f"(s4.w), "f"(sa));
    }
}

// 16-byte global -> shared copy; src_bytes = 0 writes zeros without reading.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(src_bytes)
                 : "memory");
}

// TMA tile store shared -> global (bulk-group completion), and its waits.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// at most one store group still reading its shared-memory source
__device__ __forceinline__ void bulk_wait_read_1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// every store group complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// generic-proxy writes to shared memory become visible to the TMA (async proxy)
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Wait for this thread's outstanding TMEM loads.  The registers pass through
// the asm as read-write operands, so no use of them can move above the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]) :: "memory");
}
// Orders a second load's registers after a preceding tmem_ld_wait.
__device__ __forceinline__ void reg_after_wait(uint32_t (&r)[32]) {
    asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}


// ------------------------------------------------------------ host side
// 2-D tensor [rows, cols] of `elem_bytes`-byte elements (cols contiguous;
// 1 = E4M3 codes, 2 = bf16, 4 = float32), box [box_rows, box_cols], 128-byte
// swizzle (box_cols * elem_bytes == 128).
int make_map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, int elem_bytes,
                uint32_t box_rows, uint32_t box_cols);

}  // namespace tc
}  // namespace moe
