// Dispatch layout: a deterministic, stable counting sort of the T*K
// (token, slot) selections by expert.
//
// Source: "官方揭秘DeepSeek-V3模型训练全流程" (youleyou.com), §2.2: no token
// is dropped in training or inference, so there is no capacity limit and
// every selection gets a row.  Rows of one expert are ordered by ascending
// token, which makes the layout unique.
//
// Three kernels over chunks of 64 tokens (one block for at most 1024
// selections, permute_small_kernel):
//   hist:    per-chunk histogram of expert ids (shared-memory atomics),
//   scan:    per-expert totals, exclusive scan -> offsets, and each chunk's
//            first row per expert,
//   scatter: the chunk's selections in (token, slot) order are split into
//            eight runs, one per warp; each warp's rows per expert start after
//            the earlier warps', and within a run the lanes holding the same
//            expert are ranked by lane.
#include "common.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) hist_kernel(const int32_t* __restrict__ idx, int T, int K,
                                                   int E, int32_t* __restrict__ hist,
                                                   int32_t* status) {
    extern __shared__ int32_t h[];
    griddep_wait();
    griddep_launch();
    for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
    __syncthreads();
    const int t0 = blockIdx.x * kPermuteChunk;
    const int t1 = min(T, t0 + kPermuteChunk);
    for (int p = t0 * K + threadIdx.x; p < t1 * K; p += blockDim.x) {
        const int e = idx[p];
        if (e >= 0 && e < E)
            atomicAdd(&h[e], 1);
        else
            flag_status(status, MOE_ERR_BAD_INDEX);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = h[e];
}

// One block of 1024 threads.  base[b][e] = offsets[e] + sum_{b' < b} hist[b'][e].
// Optionally writes the grouped-GEMM group offsets: E routed groups, then S
// shared groups of T rows each after the T*K routed rows (E+S+1 entries).
__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* __restrict__ hist, int nchunks,
                                                    int E, int T, int K, int S,
                                                    int32_t* __restrict__ base,
                                                    int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ go_ext) {
    __shared__ int32_t warp_sums[32];
    griddep_wait();
    griddep_launch();
    const int tid = threadIdx.x;
    int total = 0;
    if (tid < E)
        for (int b = 0; b < nchunks; ++b) total += hist[(size_t)b * E + tid];
    // block-wide exclusive scan of `total` over tid
    int v = total;
    const int lane = tid & 31, w = tid >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    if (lane == 31) warp_sums[w] = v;
    __syncthreads();
    if (w == 0) {
        int ws = warp_sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, ws, off);
            if (lane >= off) ws += o;
        }
        warp_sums[lane] = ws;
    }
    __syncthreads();
    const int excl = v - total + (w > 0 ? warp_sums[w - 1] : 0);
    if (tid < E) {
        offsets[tid] = excl;
        if (go_ext) go_ext[tid] = excl;
        if (tid == E - 1) {
            offsets[E] = excl + total;
            if (go_ext)
                for (int s = 0; s <= S; ++s) go_ext[E + s] = T * K + s * T;
        }
        int run = excl;
        for (int b = 0; b < nchunks; ++b) {
            base[(size_t)b * E + tid] = run;
            run += hist[(size_t)b * E + tid];
        }
    }
}

// Also writes the rows of the S shared-expert groups: row T*K + s*T + t is
// token t.  The chunk's selections, in (token, slot) order, are cut into
// eight consecutive runs, one per warp.  Each warp counts its run's experts;
// the counts are turned into each warp's first row per expert (the chunk's
// base plus the earlier warps' counts, one thread per expert); then each warp
// walks its run 32 selections at a time, the lanes holding the same expert
// ranked by lane (__match_any_sync), and advances its rows by their number.
// Rows of one expert thus ascend in selection order, as the layout requires.
constexpr int SCAT_WARPS = 8;
__global__ void __launch_bounds__(SCAT_WARPS * 32) scatter_kernel(const int32_t* __restrict__ idx, int T,
                                                      int K, int E, int S,
                                                      const int32_t* __restrict__ base,
                                                      int32_t* __restrict__ perm,
                                                      int32_t* __restrict__ inv_row) {
    extern __shared__ int32_t smem_scat[];
    int32_t* sel = smem_scat;                        // [kPermuteChunk * K] the chunk's selections
    int32_t* wrow = smem_scat + kPermuteChunk * K;   // [SCAT_WARPS][E] counts, then first rows
    griddep_wait();
    griddep_launch();
    const int t0 = blockIdx.x * kPermuteChunk;
    const int t1 = min(T, t0 + kPermuteChunk);
    const int n = (t1 - t0) * K;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int p = threadIdx.x; p < S * (t1 - t0); p += blockDim.x) {
        const int s = p / (t1 - t0), t = t0 + p % (t1 - t0);
        perm[(size_t)T * K + (size_t)s * T + t] = t;
    }
    for (int p = threadIdx.x; p < n; p += blockDim.x) sel[p] = idx[(size_t)t0 * K + p];
    for (int i = threadIdx.x; i < SCAT_WARPS * E; i += blockDim.x) wrow[i] = 0;
    __syncthreads();
    // this warp's run of selections: [p0, p1), whole steps of 32 lanes
    const int per = ((n + SCAT_WARPS - 1) / SCAT_WARPS + 31) / 32 * 32;
    const int p0 = min(n, warp * per), p1 = min(n, p0 + per);
    int32_t* myrow = wrow + warp * E;
    for (int p = p0 + lane; p < p1; p += 32) {
        const int e = sel[p];
        if (e >= 0 && e < E) atomicAdd(&myrow[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = base[(size_t)blockIdx.x * E + e];
        for (int w = 0; w < SCAT_WARPS; ++w) {
            const int c = wrow[w * E + e];
            wrow[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    for (int q0 = p0; q0 < p1; q0 += 32) {
        const int p = q0 + lane;
        const bool have = p < p1;
        const int e = have ? sel[p] : -1;
        const bool ok = have && e >= 0 && e < E;
        const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (ok) {
            const int row = myrow[e] + rank;
            perm[row] = t0 + p / K;
            inv_row[(size_t)t0 * K + p] = row;
        }
        __syncwarp();
        // the lowest lane of each expert's peers advances that expert's rows
        if (ok && rank == 0) myrow[e] += __popc(peers);
        __syncwarp();
    }
}

// Few selections (T*K <= 1024, E <= 1024): the whole counting sort in one
// block of 1024 threads -- thread p owns selection p, in (token, slot) order.
// Counts by shared-memory atomics, exclusive scan over the experts, then the
// 32 warps take turns in order: within a warp, the lanes holding the same
// expert are ranked by lane (match), and the expert's running row advances by
// their number, so rows of one expert ascend by token as in the three-kernel
// form (same layout, bit for bit).
constexpr int kSmallPermute = 1024;
__global__ void __launch_bounds__(kSmallPermute) permute_small_kernel(
    const int32_t* __restrict__ idx, int T, int K, int E, int S, int32_t* __restrict__ offsets,
    int32_t* __restrict__ go_ext, int32_t* __restrict__ perm, int32_t* __restrict__ inv_row,
    int32_t* status) {
    __shared__ int32_t cnt[kMaxExperts];
    __shared__ int32_t run[kMaxExperts];
    __shared__ int32_t warp_sums[32];
    griddep_wait();
    griddep_launch();
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int n = T * K;
    for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    int e_mine = -1;
    if (tid < n) {
        const int e = idx[tid];
        if (e >= 0 && e < E) {
            e_mine = e;
            atomicAdd(&cnt[e], 1);
        } else {
            flag_status(status, MOE_ERR_BAD_INDEX);
        }
    }
    __syncthreads();
    // exclusive scan of cnt over the experts (thread e holds expert e)
    const int total = tid < E ? cnt[tid] : 0;
    int v = total;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    if (lane == 31) warp_sums[w] = v;
    __syncthreads();
    if (w == 0) {
        int ws = warp_sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, ws, off);
            if (lane >= off) ws += o;
        }
        warp_sums[lane] = ws;
    }
    __syncthreads();
    if (tid < E) {
        const int excl = v - total + (w > 0 ? warp_sums[w - 1] : 0);
        offsets[tid] = excl;
        run[tid] = excl;
        if (go_ext) go_ext[tid] = excl;
        if (tid == E - 1) {
            offsets[E] = excl + total;
            if (go_ext)
                for (int s = 0; s <= S; ++s) go_ext[E + s] = T * K + s * T;
        }
    }
    for (int p = tid; p < S * T; p += blockDim.x) perm[(size_t)T * K + p] = p % T;
    __syncthreads();
    // rows in selection order, one warp at a time
    const int nwarps = (n + 31) / 32;
    for (int turn = 0; turn < nwarps; ++turn) {
        if (w == turn) {
            const unsigned same = __match_any_sync(0xffffffffu, e_mine);
            const int rank = __popc(same & ((1u << lane) - 1u));
            if (e_mine >= 0) {
                const int row = run[e_mine] + rank;
                perm[row] = tid / K;
                inv_row[tid] = row;
            }
            __syncwarp();
            if (e_mine >= 0 && rank == 0) run[e_mine] += __popc(same);
        }
        __syncthreads();
    }
}

}  // namespace

int launch_permute(const int32_t* idx, int T, int K, int E, int32_t* offsets, int32_t* perm,
                   int32_t* inv_row, int32_t* go_ext, int S, int32_t* status,
                   int32_t* ws_hist, int32_t* ws_base, cudaStream_t st) {
    const int nchunks = (T + kPermuteChunk - 1) / kPermuteChunk;
    int rc;
    if (T > 0 && (long long)T * K <= kSmallPermute && E <= kMaxExperts)
        return launch_pdl(permute_small_kernel, dim3(1), dim3(kSmallPermute), 0, st, idx, T, K, E, S,
                          offsets, go_ext, perm, inv_row, status);
    if (nchunks > 0 && (rc = launch_pdl(hist_kernel, dim3(nchunks), dim3(256), sizeof(int32_t) * E,
                                        st, idx, T, K, E, ws_hist, status)))
        return rc;
    if ((rc = launch_pdl(scan_kernel, dim3(1), dim3(1024), 0, st, (const int32_t*)ws_hist, nchunks,
                         E, T, K, S, ws_base, offsets, go_ext)))
        return rc;
    if (nchunks > 0)
        rc = launch_pdl(scatter_kernel, dim3(nchunks), dim3(SCAT_WARPS * 32),
                        sizeof(int32_t) * ((size_t)kPermuteChunk * K + (size_t)SCAT_WARPS * E), st,
                        idx, T, K, E, S, (const int32_t*)ws_base, perm, inv_row);
    return rc;
}

}  // namespace moe
