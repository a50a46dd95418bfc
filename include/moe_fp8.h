/*
 * moe_fp8.h -- C ABI of libmoefp8.so: the forward pass of one DeepSeekMoE
 * layer with auxiliary-loss-free routing and fine-grained FP8 expert GEMMs,
 * written for NVIDIA B300 (sm_103a).
 *
 * Sources (web pages summarising the DeepSeek-V3 technical report):
 *   [TH]  "รายงานเชิงเทคนิคของ DeepSeek-V3" (xyznot.com/th/paper/2412.19437),
 *         Method §2 (equations for h'_t, s_{i,t}, g'_{i,t}; bias update) and
 *         Key ideas, FP8 bullet (E4M3, 1x128 / 128x128 scaling, FP32
 *         promotion every N_c = 128).
 *   [YLY] "官方揭秘DeepSeek-V3模型训练全流程" (youleyou.com), §2.2
 *         (no token dropping) and §4.3 FP8 训练.
 *   [DB]  "Deepseek V3 国货之光 开源之光" (databean.com.cn), section
 *         "Auxiliary-Loss-Free Load Balancing".
 *
 * Conventions shared by every call:
 *   - Tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates device memory, never frees, and keeps no pointer after
 *     a call returns.  Scratch comes from a caller-provided workspace.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     only enqueue work; they do not synchronise, except
 *     moe_check_device_status, which says so.
 *   - Types: bf16 = uint16_t bit pattern of bfloat16; fp8 = uint8_t code of
 *     OCP FP8 E4M3FN (max 448, no infinities).  Layouts are row-major.
 *   - Every call returns an int status (enum moe_status).  Arguments are
 *     validated on the host before anything is enqueued; on a non-zero
 *     status nothing was enqueued, except MOE_ERR_CUDA, which reports a
 *     failed launch (moe_last_cuda_error() gives the cudaError_t of the
 *     calling thread).  No call aborts or throws.
 *   - Activation scales are stored "MN-major": scale of row r and K-block kb
 *     at scales[kb * scale_ld + r].  Weight scales are per 128x128 block:
 *     for a [G, N, K] weight stack, scale of group g, row block nb, column
 *     block kb at scales[(g * (N/128) + nb) * (K/128) + kb].
 */
#ifndef MOE_FP8_H
#define MOE_FP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,       /* null pointer, K > E, K > 32, E > 1024, negative size, ... */
    MOE_ERR_UNSUPPORTED_SHAPE = -2, /* d or I not a multiple of 128, too many groups, ...        */
    MOE_ERR_MISALIGNED = -3,        /* a pointer is not 16-byte aligned                           */
    MOE_ERR_CUDA = -4,              /* a CUDA call failed; see moe_last_cuda_error()              */
    MOE_ERR_TIMEOUT = -5,           /* a GEMM pipeline wait ran out (device status word)          */
    MOE_ERR_WORKSPACE = -6,         /* workspace too small                                        */
    MOE_ERR_BAD_INDEX = -7          /* device data held an index out of range (device status)     */
};

/* Grouped GEMM modes (moe_grouped_gemm_fp8). */
enum moe_gemm_mode {
    MOE_GEMM_GATE_UP_SILU_QUANT = 1, /* h = SiLU(A W_gate^T) * (A W_up^T), re-quantised 1x128 */
    MOE_GEMM_DOWN = 2,               /* y = A W_down^T, stored as bf16                         */
    MOE_GEMM_GATE_UP_DGRAD = 3,      /* [dG | dU] from recomputed G, U and dH (moe_backward_dgrad) */
    MOE_GEMM_DOWN_F32 = 4            /* y = A W_down^T, stored as float32                      */
};

/* One DeepSeekMoE layer: d hidden, E routed experts (top-K of them per
 * token), S shared experts, expert intermediate size I.  Weight stacks hold
 * the E routed experts first and the S shared experts after them.
 * Limits checked by every call that takes a layer: 1 <= K <= min(E, 32),
 * E <= 1024, E + S <= 1088, K + S <= 32 (a token has at most 32 dispatch
 * rows), d and I multiples of 128. */
typedef struct moe_layer_t {
    int d, E, K, S, I;
    const float* centroids;   /* [E, d] expert centroids e_i                          */
    const float* bias;        /* [E] selection bias b_i (moe_update_bias changes it)  */
    const uint8_t* w_gate;    /* [E+S, I, d] fp8                                      */
    const uint8_t* w_up;      /* [E+S, I, d] fp8                                      */
    const uint8_t* w_down;    /* [E+S, d, I] fp8                                      */
    const float* s_gate;      /* [E+S, I/128, d/128] block scales                     */
    const float* s_up;        /* [E+S, I/128, d/128]                                  */
    const float* s_down;      /* [E+S, d/128, I/128]                                  */
    /* Group-limited routing (moe_route_grouped); n_groups = 0: plain top-K.  */
    int n_groups, topk_groups, group_topk;
} moe_layer_t;

/* Text of a status code (static storage; never NULL). */
const char* moe_status_string(int status);

/* cudaError_t of the last failed CUDA call made by the calling thread. */
int moe_last_cuda_error(void);

/* Number of kernels this process has launched through the library. */
uint64_t moe_kernel_launches(void);

/* Limit, in SM clock cycles, of every wait inside the grouped GEMMs'
 * pipelines (a stage of operands, a TMEM buffer, a slot of scales, the next
 * tile) for the launches made after this call, by any thread; cycles <= 0
 * restores the default of 4e9 (about 2 s).  A wait that runs out records
 * MOE_ERR_TIMEOUT in the call's status word; the kernel then stops, waits
 * (with the long limit) for its copies and MMAs in flight, releases its
 * tensor memory and returns, so the context stays usable.  Returns the
 * previous limit.  A diagnostic of the failure path (no counterpart in the
 * pages): a limit of a few hundred cycles makes the first wait run out. */
long long moe_set_pipeline_wait_limit(long long cycles);

/* Test switch of the same failure path (no counterpart in the pages): with
 * on != 0 the grouped GEMMs launched afterwards issue no operand loads, so
 * their first pipeline waits run out after the wait limit and the calls
 * report MOE_ERR_TIMEOUT in their status word; on = 0 restores normal
 * operation.  Returns the previous setting.  Only for tests of the timeout
 * path; results of the affected calls are incomplete. */
int moe_set_pipeline_stall(int on);

/* Workspace bytes moe_forward needs for up to T_max tokens of layer L
 * (0 if L is invalid).  The same workspace serves moe_route and
 * moe_permute at the same T. */
size_t moe_workspace_size(const moe_layer_t* L, int T_max);

/* Online 1x128 activation quantisation ([TH] Key ideas, FP8 bullet;
 * [YLY] §4.3: online max-abs per 1x128 tile).  Output row r takes input row
 * gather_rows[r] (or r when gather_rows is NULL; rows whose index is outside
 * [0, n_src) are skipped and flagged MOE_ERR_BAD_INDEX in *status when status
 * is not NULL).  Per tile: amax = max |x|; scale = amax / 448 (IEEE float32
 * division); q = E4M3(x / scale) rounded to nearest even and saturated; a
 * tile with amax = 0 gets scale 1 and all codes 0.
 *   x [n_src, d] bf16;  q [M, d] fp8;  scales at scales[kb * scale_ld + r],
 *   scale_ld >= M.  d must be a multiple of 128; x, q 16-byte aligned. */
int moe_quant_1x128(const uint16_t* x, int n_src, const int32_t* gather_rows, int M, int d,
                    uint8_t* q, float* scales, int scale_ld, int32_t* status, void* stream);

/* The dispatch-fused form of moe_quant_1x128 ([TH] Key ideas, FP8 bullet;
 * [YLY] §4.3 and §2.2): quantisation is row-local, so every token is
 * quantised once and its codes and scales are written to each row the
 * dispatch gave it -- routed rows inv_row[t, 0..K) (moe_permute) and shared
 * rows T*K + s*T + t, s < S.  Same rule and the same bits as
 * moe_quant_1x128 with gather_rows = perm_token.
 *   x [T, d] bf16; q [T*(K+S), d] fp8; scales at scales[kb * scale_ld + row],
 *   scale_ld >= T*(K+S).  1 <= K + S <= 32.  A routed row outside
 *   [0, T*(K+S)) is skipped and flagged MOE_ERR_BAD_INDEX in *status. */
int moe_quant_1x128_dispatch(const uint16_t* x, int T, int d, const int32_t* inv_row, int K,
                             int S, uint8_t* q, float* scales, int scale_ld, int32_t* status,
                             void* stream);

/* 128x128 block quantisation of a weight matrix ([TH] Key ideas, FP8 bullet;
 * [YLY] §4.3), same rounding rule as moe_quant_1x128 with one scale per
 * block.  w [R, C] float32; q [R, C] fp8; scales [R/128, C/128].  R and C
 * multiples of 128; w and q 16-byte aligned. */
int moe_quant_128x128(const float* w, int R, int C, uint8_t* q, float* scales, void* stream);

/* Router ([TH] Method §2: s_{i,t} = Sigmoid(u_t^T e_i); g'_{i,t} = s_{i,t}
 * when s_{i,t} + b_i is among the top K of {s_{j,t} + b_j}; g normalises g'.
 * [DB]: the bias steers the selection only).  For every token t:
 *   topk_idx [T, K] int32  experts by descending s + b (equal: lower index),
 *   topk_gate [T, K] float s of each selected expert over their sum,
 *   tie_flag [T] uint8     1 when the K-th and (K+1)-th biased scores differ
 *                          by less than 1e-6 (their order may depend on
 *                          rounding), else 0,
 *   counts [E] int32       selections per expert (overwritten).
 * u [T, d] bf16; centroids [E, d]; bias [E].  1 <= K <= min(E, 32),
 * E <= 1024.  The logits that decide the selection and the gates are float32
 * sums with compensation (error about one float32 rounding): every logit is
 * first estimated on the tensor cores (bf16 token row against a two-piece
 * bf16 split of the centroid), and the experts whose estimate lies within the
 * estimate's error bound of the K-th biased score are recomputed exactly.
 * Workspace: at least moe_route_workspace_size(T, d, E) bytes, 256-byte
 * aligned; its first int32 is this call's device status word (0, or
 * MOE_ERR_TIMEOUT when a bounded device wait gave up; read it with
 * moe_check_device_status(ws, stream)). */
int moe_route(const uint16_t* u, const float* centroids, const float* bias, int T, int d, int E,
              int K, int32_t* topk_idx, float* topk_gate, uint8_t* tie_flag, int32_t* counts,
              void* ws, size_t ws_bytes, void* stream);

/* Group-limited routing.  The pages say only that a token is sent to at most
 * M = 4 nodes ([YLY] §2.2; [SYH], table of innovations); the scoring is this
 * library's reading: the E experts form n_groups contiguous groups of
 * E / n_groups (one per node); a group's score is the float32 sum, largest
 * first, of its group_topk largest biased scores s + b; the topk_groups
 * groups with the largest scores are kept (equal: lower group index); then
 * the top K by s + b among the kept groups' experts, gates and counts as in
 * moe_route.  tie_flag is also 1 when the last kept and the next group score
 * differ by less than 1e-6.  1 <= n_groups <= 32, n_groups divides E,
 * 1 <= topk_groups <= n_groups, 1 <= group_topk <= E / n_groups,
 * K <= topk_groups * E / n_groups.  Same logits, workspace and status word as
 * moe_route (the experts whose scores the group choice or the selection
 * depend on are recomputed exactly). */
int moe_route_grouped(const uint16_t* u, const float* centroids, const float* bias, int T, int d,
                      int E, int K, int n_groups, int topk_groups, int group_topk,
                      int32_t* topk_idx, float* topk_gate, uint8_t* tie_flag, int32_t* counts,
                      void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes moe_route needs for T tokens, hidden size d and E experts
 * (0 for invalid sizes). */
size_t moe_route_workspace_size(int T, int d, int E);

/* Check hook for moe_route's screening step (no counterpart in the pages):
 * writes the tensor-core logit estimates l~ [T, E] float32 to logits and the
 * centroid norms used in the error bound to norms [E] float32, both device
 * memory.  moe_route treats |l~_e - l_e| <= 2^-11 |u_t| norms[e] as the
 * estimate's error bound.  Same workspace rules as moe_route. */
int moe_route_estimate_logits(const uint16_t* u, const float* centroids, int T, int d, int E,
                              float* logits, float* norms, void* ws, size_t ws_bytes,
                              void* stream);

/* moe_route without a workspace, for callers that cannot allocate device
 * memory when they route (a serving engine whose memory pool owns the whole
 * device, a runtime whose allocator is out of reach of the launching thread,
 * or code that must not allocate between two points it measures or
 * captures).  The pages have no counterpart of this call: it is a service of
 * this library, not a step of the method.  Same arguments and outputs as
 * moe_route, minus ws/ws_bytes; every logit is computed on the CUDA cores
 * with the same compensated summation (so results agree with moe_route up
 * to float32 rounding: selections may differ only on flagged near-ties, gates
 * by a few ulps).  The [T, E] logits live in a
 * fixed 4 MB array in the library's device memory, so T * E must be at most
 * 1048576 (MOE_ERR_WORKSPACE otherwise); the rest of the array holds split
 * partial sums that are added in a fixed order, so repeated calls on the
 * same input give identical results.  The first call on each device looks
 * up that array's device address (cudaGetSymbolAddress); make that first call
 * before any stream capture.  Every call shares the array: calls that
 * overlap on the GPU (other streams, other host threads) race on it.
 * Allocates nothing (no cudaMalloc, cudaFree or allocating library call). */
int moe_route_noalloc(const uint16_t* u, const float* centroids, const float* bias, int T, int d,
                      int E, int K, int32_t* topk_idx, float* topk_gate, uint8_t* tie_flag,
                      int32_t* counts, void* stream);

/* Dispatch layout ([YLY] §2.2: no token is dropped, so every (token, slot)
 * pair gets a row).  A stable counting sort of the T*K pairs by expert, plus
 * the rows of the S shared experts, which see every token:
 *   offsets [E+1]          exclusive scan of the per-expert counts,
 *   group_offsets [E+S+1]  (nullable) rows of the E routed groups followed by
 *                          S shared groups of T rows each -- the
 *                          group_offsets of moe_grouped_gemm_fp8,
 *   perm_token [T*(K+S)]   token of each row: routed rows of one expert
 *                          ascend by token; row T*K + s*T + t is token t,
 *   inv_row [T, K]         routed row of each (token, slot).
 * An expert index outside [0, E) is skipped and flagged MOE_ERR_BAD_INDEX in
 * *status (if not NULL).  Workspace: moe_workspace_size of a layer with the
 * same E and T (or at least 2 * 256-byte-rounded ceil(T/64) * E * 4 bytes),
 * 256-byte aligned. */
int moe_permute(const int32_t* topk_idx, int T, int K, int E, int S, int32_t* offsets,
                int32_t* group_offsets, int32_t* perm_token, int32_t* inv_row, int32_t* status,
                void* ws, size_t ws_bytes, void* stream);

/* Grouped block-scaled FP8 GEMM on tcgen05 tensor cores ([TH] Key ideas,
 * FP8 bullet; [YLY] §4.3: each 128-wide K slab is summed on the tensor core
 * and promoted to an FP32 accumulator with its 1x128 activation scale and
 * 128x128 weight scale: acc += partial * (sa * sw)).
 *   A [M_total, Kdim] fp8, sa [Kdim/128][M_total];
 *   group_offsets [G+1] (device): group g owns rows [go[g], go[g+1]) of A
 *   and of the output, and uses weight slice g.
 *   W0 [G, N, Kdim] fp8, sw0 [G, N/128, Kdim/128]; W1 / sw1 the same shape
 *   (GATE_UP mode only, NULL for DOWN).
 *   mode GATE_UP_SILU_QUANT: W0 = W_gate, W1 = W_up, N = I; out = h codes
 *     [M_total, N] fp8 with out_scales [N/128][M_total], where
 *     h = SiLU(A W0^T) * (A W1^T), SiLU(x) = x / (1 + exp(-x)), quantised
 *     per 1x128 tile with the moe_quant_1x128 rule.
 *   mode DOWN: W0 = W_down, N = d; out = y [M_total, N] bf16 (round to
 *     nearest even); out_scales unused.
 *   mode DOWN_F32: as DOWN with y stored as float32.
 * Rows outside every group are left untouched.  Kdim and N multiples of 128;
 * G <= 1088; all pointers 16-byte aligned.  status (device int32 [2],
 * nullable): status[0] receives MOE_ERR_TIMEOUT if a pipeline wait ran out
 * (the kernel then stops early and its output is incomplete); status[1] is
 * the call's tile counter (cleared by the call).  Each CTA's first output
 * tile is the one numbered like the CTA; the later tiles are claimed from the
 * counter in order, so tiles that share a weight panel run together.
 * Without a status buffer every CTA takes every grid-th tile. */
int moe_grouped_gemm_fp8(int mode, const uint8_t* A, const float* sa, int M_total,
                         const int32_t* group_offsets, int G, const uint8_t* W0,
                         const uint8_t* W1, const float* sw0, const float* sw1, int N, int Kdim,
                         void* out, float* out_scales, int32_t* status, void* stream);

/* moe_grouped_gemm_fp8 for groups with few rows (decode batches; modes
 * GATE_UP_SILU_QUANT and DOWN): same arguments, arithmetic and results, with
 * tiles of 128 weight rows by up to 32 rows of a group (the weight block on
 * the tensor core's M side, the rows on its N side).  A group's rows are cut
 * into chunks of 32, each a tile of its own, so a group with many rows (a hot
 * expert) is spread over as many CTAs; the chunks of one weight panel are
 * claimed together and read the panel from HBM once.  moe_forward uses it
 * for the gate/up GEMM of batches of at most 64 tokens and for the down
 * GEMM of batches of at most 4. */
int moe_grouped_gemm_fp8_small(int mode, const uint8_t* A, const float* sa, int M_total,
                               const int32_t* group_offsets, int G, const uint8_t* W0,
                               const uint8_t* W1, const float* sw0, const float* sw1, int N,
                               int Kdim, void* out, float* out_scales, int32_t* status,
                               void* stream);

/* The layer's down projection (moe_grouped_gemm_fp8 in DOWN mode, same
 * arithmetic) with its outputs split by precision: the rows of groups
 * [0, f32_group0) go to y [*, N] as bf16, the rows of groups
 * [f32_group0, G) to y_f32 [*, N] as float32 at row (row - f32_row0).  The
 * layer passes f32_group0 = E and f32_row0 = T*K: routed outputs in bf16,
 * shared outputs (rows T*K ...) in float32.  small_tiles != 0 selects the
 * tiles of moe_grouped_gemm_fp8_small.  H [M_total, Kdim] fp8 with sh
 * [Kdim/128][M_total]; W [G, N, Kdim] fp8 with sw [G, N/128, Kdim/128];
 * status as in moe_grouped_gemm_fp8. */
int moe_grouped_gemm_fp8_down(const uint8_t* H, const float* sh, int M_total,
                              const int32_t* group_offsets, int G, int f32_group0, int f32_row0,
                              const uint8_t* W, const float* sw, int N, int Kdim, uint16_t* y,
                              float* y_f32, int small_tiles, int32_t* status, void* stream);

/* Combine ([TH] Method §2: h'_t = u_t + sum_s FFN_s(u_t) + sum_i g_{i,t}
 * FFN_i(u_t)).  h_out[t] = u[t] + sum_s Y_shared[s*T + t] +
 * sum_k topk_gate[t,k] * Y[inv_row[t,k]], summed in float32.
 *   u [T, d] bf16; Y [*, d] bf16 (routed rows); Y_shared [S*T, d] float32
 *   (the shared experts' outputs, which enter h' with weight 1, are kept in
 *   float32; the bf16 rounding of the routed outputs is averaged by gates
 *   that sum to 1; may be NULL when S = 0); h_out [T, d] float32 (the rows of
 *   moe_grouped_gemm_fp8_down).  d multiple of 8; pointers 16-byte aligned. */
int moe_combine(const uint16_t* u, const uint16_t* Y, const float* topk_gate,
                const int32_t* inv_row, const float* Y_shared, int T, int d, int K, int S,
                float* h_out, void* stream);

/* The whole layer forward: route, dispatch, quantise, GEMM (gate/up + SiLU),
 * GEMM (down), combine -- all enqueued on `stream` with no host sync.
 * Outputs: h_out [T, d] float32 and the routing (topk_idx, topk_gate,
 * counts, tie_flag as in moe_route, or moe_route_grouped when L->n_groups >
 * 0), which moe_update_bias consumes.  Below 256 tokens without group
 * limits the logits are all summed exactly on CUDA cores (the router of
 * moe_route_noalloc, with partial sums added in a fixed order) instead of
 * the tensor-core screen: the same selection rule and tie flag; only tokens
 * flagged as near ties may select differently from moe_route.  Repeated
 * calls on the same input give identical results.
 * ws: at least moe_workspace_size(L, T) bytes, 256-byte aligned.  Its first
 * 16 bytes hold the device status word of this call (read it with
 * moe_check_device_status(ws, stream)). */
int moe_forward(const moe_layer_t* L, const uint16_t* u, int T, float* h_out, int32_t* topk_idx,
                float* topk_gate, int32_t* counts, uint8_t* tie_flag, void* ws, size_t ws_bytes,
                void* stream);

/* Device buffers of one batch in flight for moe_forward_host (caller-owned,
 * device memory): u [T, d] bf16, h [T, d] float32 (16-byte aligned),
 * topk_idx [T, K] int32, topk_gate [T, K] float32, tie_flag [T] uint8,
 * counts [E] int32. */
typedef struct moe_batch_buffers_t {
    uint16_t* u;
    float* h;
    int32_t* topk_idx;
    float* topk_gate;
    uint8_t* tie_flag;
    int32_t* counts;
} moe_batch_buffers_t;

/* The layer over a sequence of n_batches batches of T tokens held in host
 * memory (page-locked, so the copies run asynchronously): for batch k,
 * u_host[k] [T, d] bf16 goes to buf[k % 2].u on h2d_stream, moe_forward runs
 * on compute_stream, then -- when gamma != 0 -- moe_update_bias with that
 * batch's counts (the next batch is routed with the updated bias), and
 * buf[k % 2].h goes back to h_host[k] [T, d] float32 on d2h_stream.  Events
 * (created and released by the call) order the three streams so that the
 * upload of batch k+1 and the download of batch k-1 overlap the compute of
 * batch k; the batches share ws (moe_workspace_size(L, T) bytes, 256-byte
 * aligned), whose status word is cleared once and then collects every
 * batch's device errors.  Nothing synchronises the host: synchronise
 * d2h_stream before reading h_host.  With the same stream passed three times
 * the batches run one after another.  The pages describe no host interface;
 * this is a service of the library for inputs that arrive from the host. */
int moe_forward_host(const moe_layer_t* L, int T, int n_batches, const uint16_t* const* u_host,
                     float* const* h_host, float gamma, const moe_batch_buffers_t* buf, void* ws,
                     size_t ws_bytes, void* compute_stream, void* h2d_stream, void* d2h_stream);

/* Two micro-batches in flight on one GPU ([YLY] §4.4 inference deployment:
 * the computation of one micro-batch overlaps the dispatch and combine work
 * of the other).  The layer over n_batches device-resident batches of T
 * tokens (batches[k].u in, batches[k].h and the routing out, as moe_forward),
 * with the bias stepped by moe_update_bias after each batch when gamma != 0.
 * Batch k's routing, dispatch and quantisation (side_stream) run while batch
 * k-1's expert GEMMs run (gemm_stream), and batch k-1's combine while batch
 * k's GEMMs run; the GEMMs' persistent grids leave reserve_sms SMs free for
 * the side stream's kernels (0: the GEMMs take every SM and the side work
 * only fills the gaps).  ws0 and ws1 (moe_workspace_size(L, T) bytes each,
 * 256-byte aligned) alternate between the batches; each one's status word
 * collects its batches' device errors.  Results are bit-identical to
 * moe_forward + moe_update_bias batch after batch.  Nothing synchronises
 * the host: synchronise side_stream (it holds the last combine) before
 * reading the outputs. */
int moe_forward_pipelined(const moe_layer_t* L, int T, int n_batches,
                          const moe_batch_buffers_t* batches, float gamma, void* ws0, void* ws1,
                          size_t ws_bytes, int reserve_sms, void* gemm_stream, void* side_stream);

/* Input gradient of the layer (the pages: FP8 also carries part of the
 * gradient propagation, [SYH] FP8 資料格式訓練; they wish for transposed
 * GEMMs in hardware, [YLY] hardware suggestions).  Reading: every expert
 * backward GEMM follows the forward's FP8 rule.  The transposed weights are
 * exact in FP8 with 128x128 block scales (codes moved, each block keeps its
 * scale); moe_prepare_backward_weights writes them once per weight update:
 *   w_down_t [E+S, I, d] fp8 with s_down_t [E+S, I/128, d/128],
 *   w_gu_t   [E+S, d, 2I] fp8 = [W_gate^T | W_up^T] with s_gu_t [E+S, d/128, 2I/128]. */
typedef struct moe_layer_bwd_t {
    const uint8_t* w_down_t;
    const float* s_down_t;
    const uint8_t* w_gu_t;
    const float* s_gu_t;
} moe_layer_bwd_t;

int moe_prepare_backward_weights(const moe_layer_t* L, uint8_t* w_down_t, float* s_down_t,
                                 uint8_t* w_gu_t, float* s_gu_t, void* stream);

/* Workspace bytes moe_backward_dgrad needs for up to T_max tokens (0 if L is
 * invalid); its first 16 bytes hold the call's device status word. */
size_t moe_backward_workspace_size(const moe_layer_t* L, int T_max);

/* du = d loss / d u for a forward that has just run: call after moe_forward
 * with the same L, u and T, and pass that call's workspace (fwd_ws; its
 * dispatched activations, group offsets, dispatch rows and expert outputs
 * are read) and routing (topk_idx, topk_gate).  dh [T, d] bf16 is the
 * gradient of h'; du [T, d] float32.  Steps: the gradient of each dispatch
 * row (g_k dh routed, dh shared; float32 product) quantised per 1x128 tile;
 * dH = bf16(dy W_down); G and U recomputed by the gate/up GEMM, whose
 * epilogue forms dG = dH U sigma (1 + G (1 - sigma)), dU = dH G sigma
 * (sigma = 1 / (1 + e^-G)) and quantises [dG | dU] per 1x128 tile;
 * dA = bf16([dG | dU] [W_gate ; W_up]); du = dh + the token's rows of dA, plus
 * the gates' dependence on u: with dg_k = dh . y_k, s_k = sigmoid(u . e_k)
 * (exact logit, as moe_route) and S = sum s_k,
 * du += sum_k (dg_k - sum_j g_j dg_j) / S * s_k (1 - s_k) e_k.  The bias has no
 * gradient.  bwd_ws: moe_backward_workspace_size(L, T) bytes, 256-byte
 * aligned; moe_check_device_status(bwd_ws, stream) reads its status. */
int moe_backward_dgrad(const moe_layer_t* L, const moe_layer_bwd_t* B, const uint16_t* u,
                       const uint16_t* dh, int T, const int32_t* topk_idx, const float* topk_gate,
                       float* du, void* fwd_ws, size_t fwd_ws_bytes, void* bwd_ws,
                       size_t bwd_ws_bytes, void* stream);

/* Weight gradients (the pages keep FP8 activations in storage and master
 * weights and gradients in 16/32 bits, [SYH] FP8 資料格式訓練 and [YLY]
 * §4.3; they wish for transposed GEMMs in hardware, [YLY] hardware
 * suggestions, because tensors held in 1x128 tiles along features are
 * contracted over tokens here).  Reading: each FP8 tensor the layer holds is
 * dequantised (x = dec(q) * s, a float32 product), transposed and
 * re-quantised in 128x1 tiles: 128 consecutive rows of one group by one
 * column, scale = amax / 448, code = E4M3(x / scale) (the moe_quant_1x128
 * rule); a group's last block is ragged and a block never spans two groups.
 *
 * Padded layout of a transposed operand with C columns: slab offsets pb[g] =
 * sum over g' < g of ceil(rows_g' / 128); group g's rows become columns
 * 128 pb[g] .. of qt [C, ld] (codes past the group's last row are 0), and
 * the scales st [ld/128, C] hold slab j's C scales contiguously.  ld must be
 * at least moe_wgrad_ld(M, G) (a multiple of 128 covering any row split). */
int moe_wgrad_ld(int M, int G);

/* q [M, C] E4M3 codes with scales [C/128][M] (the 1x128 layout of
 * moe_quant_1x128); group_offsets [G+1] (device) as in moe_grouped_gemm_fp8
 * (non-decreasing, within [0, M]; otherwise MOE_ERR_BAD_INDEX goes to
 * status[0] and nothing is written).  Writes qt [C, ld] and st [ld/128, C]
 * in the padded layout above; columns past the last group's block are not
 * written.  C a multiple of 128; q, qt 16-byte aligned. */
int moe_requant_128x1(const uint8_t* q, const float* scales, int M, int C,
                      const int32_t* group_offsets, int G, uint8_t* qt, float* st, int ld,
                      int32_t* status, void* stream);

/* Token-contracted FP8 GEMM of the weight gradient: for every group g,
 *   out_g[n, m] = sum over g's slabs kb of fma(p, sA[kb, n] * sB[kb, m], .)
 * in float32 (p = the tensor-core sum of the slab's 128 rows; the scale
 * product is a float32 multiply), i.e. out_g = At_g Bt_g^T over g's rows.
 *   At [Na, ld], sAt [ld/128, Na]; Bt [Nb, ld], sBt [ld/128, Nb] (padded
 *   layout of moe_requant_128x1 with the same group_offsets).
 *   Output rows n < split go to out0 [G, split, Nb], rows n >= split to
 *   out1 [G, Na - split, Nb] (NULL when split == Na).  A group without rows
 *   gets zeros.  Na, Nb, split multiples of 128 (0 < split <= Na); ld a
 *   multiple of 16 covering the padded rows; out pointers 16-byte aligned.
 * status (device int32 [2], nullable) as in moe_grouped_gemm_fp8. */
int moe_wgrad_gemm_fp8(const uint8_t* At, const float* sAt, int Na, const uint8_t* Bt,
                       const float* sBt, int Nb, int ld, const int32_t* group_offsets, int G,
                       float* out0, float* out1, int split, int32_t* status, void* stream);

/* Workspace bytes moe_backward_wgrad needs for up to T_max tokens (the four
 * re-quantised operands; 0 if L is invalid). */
size_t moe_wgrad_workspace_size(const moe_layer_t* L, int T_max);

/* Weight gradients of every expert for the batch of the last moe_forward and
 * moe_backward_dgrad calls (same L and T; their workspaces are read: the
 * forward's activation rows A and h, the backward's dy and [dG | dU]).  The
 * four tensors are re-quantised in 128x1 tiles into wgrad_ws, then
 *   dW_down [E+S, d, I] = dy^T h   and   [dW_gate ; dW_up] [E+S, 2I, d] =
 *   [dG | dU]^T A, both float32, written (not accumulated).
 * Experts that no token selected get zeros.  Device errors go to the status
 * word of bwd_ws (moe_check_device_status(bwd_ws, stream)).  wgrad_ws:
 * moe_wgrad_workspace_size(L, T) bytes, 256-byte aligned. */
int moe_backward_wgrad(const moe_layer_t* L, int T, float* dW_gate, float* dW_up, float* dW_down,
                       void* fwd_ws, size_t fwd_ws_bytes, void* bwd_ws, size_t bwd_ws_bytes,
                       void* wgrad_ws, size_t wgrad_ws_bytes, void* stream);

/* Auxiliary-loss-free bias update at the end of a step ([TH] Method §2:
 * b_i -= gamma when expert i is overloaded, += gamma when underloaded;
 * gamma = 0.001 there).  With n = T*K selections, expert e is overloaded when
 * counts[e] * E > n and underloaded when counts[e] * E < n; equal load keeps
 * b_e.  bias [E] float32 is updated in place. */
int moe_update_bias(const int32_t* counts, int E, int T, int K, float gamma, float* bias,
                    void* stream);

/* Waits for `stream`, reads the device status word at `status` (written by
 * moe_quant_1x128, moe_permute, moe_grouped_gemm_fp8 or moe_forward) and
 * returns it (MOE_OK when nothing was flagged), then clears it. */
int moe_check_device_status(int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FP8_H */
