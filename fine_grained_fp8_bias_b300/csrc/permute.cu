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
//   scatter: each thread owns an expert and walks the chunk's selections in
//            (token, slot) order, handing out consecutive rows.
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
// token t.
__global__ void __launch_bounds__(256) scatter_kernel(const int32_t* __restrict__ idx, int T,
                                                      int K, int E, int S,
                                                      const int32_t* __restrict__ base,
                                                      int32_t* __restrict__ perm,
                                                      int32_t* __restrict__ inv_row) {
    extern __shared__ int32_t sel[];            // this chunk's selections, (token, slot) order
    griddep_wait();
    griddep_launch();
    const int t0 = blockIdx.x * kPermuteChunk;
    const int t1 = min(T, t0 + kPermuteChunk);
    const int n = (t1 - t0) * K;
    for (int p = threadIdx.x; p < S * (t1 - t0); p += blockDim.x) {
        const int s = p / (t1 - t0), t = t0 + p % (t1 - t0);
        perm[(size_t)T * K + (size_t)s * T + t] = t;
    }
    for (int p = threadIdx.x; p < n; p += blockDim.x) sel[p] = idx[(size_t)t0 * K + p];
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int row = base[(size_t)blockIdx.x * E + e];
        for (int p = 0; p < n; ++p) {
            if (sel[p] == e) {
                const int t = t0 + p / K;
                perm[row] = t;
                inv_row[(size_t)t0 * K + p] = row;
                ++row;
            }
        }
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
        rc = launch_pdl(scatter_kernel, dim3(nchunks), dim3(256),
                        sizeof(int32_t) * kPermuteChunk * K, st, idx, T, K, E, S,
                        (const int32_t*)ws_base, perm, inv_row);
    return rc;
}

}  // namespace moe
