/*
 * Plain CPU oracle of the DeepSeekMoE FP8 layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file (through oracle/oracle.py).  The CUDA
 * library never includes, links or calls it, and the two share no code.
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -shared -fPIC -lm.
 *
 * Every step is written out the plain way, in the order the pages give it,
 * single-threaded and slow on purpose.  Sources (web pages summarising the
 * DeepSeek-V3 technical report):
 *   [TH]  "รายงานเชิงเทคนิคของ DeepSeek-V3" (xyznot.com/th/paper/2412.19437):
 *         Method §2 "DeepSeekMoE with auxiliary-loss-free balancing" -- the
 *         equations for h'_t, s_{i,t} and g'_{i,t}, and the bias update rule;
 *         Key ideas, FP8 bullet -- E4M3 on all tensors, 1x128 activation
 *         tiles, 128x128 weight blocks, promotion to FP32 every N_c = 128.
 *   [YLY] "官方揭秘DeepSeek-V3模型训练全流程" (youleyou.com): §2.2 DeepSeekMoE
 *         (no token dropping); §4.3 FP8 训练 (fine-grained quantisation,
 *         increased accumulation precision, online max-abs quantisation).
 *   [DB]  "Deepseek V3 国货之光 开源之光" (databean.com.cn): section
 *         "Auxiliary-Loss-Free Load Balancing" (the bias only steers top-K;
 *         gates are the normalised unbiased scores).
 *   [SYH] "DeepSeek V3技術報告" (sheng-yao-huang.com): section "FP8 資料格式
 *         訓練", item 1 (map the block max to the format max).
 *
 * Readings taken where the pages leave a step open (each one is a choice,
 * not something the pages print):
 *   R1  E4M3 is OCP FP8 E4M3FN; encoding rounds to nearest, ties to even,
 *       and saturates to +-448.
 *   R2  tile scale = amax / 448 (float32 division); code = enc(x / scale)
 *       (float32 division, then R1); a tile with amax = 0 gets scale 1.0 and
 *       all codes 0x00.
 *   R3  logits accumulate in double and round once to float; sigmoid is
 *       evaluated in double and rounded to float; the biased score z = s + b
 *       is a float32 add.
 *   R4  top-K orders by descending z; equal z: lower expert index first.
 *       A token is flagged "near tie" when z_(K) - z_(K+1) < 1e-6.
 *   R5  gate g_k = s_k / sum of the selected s (sum and quotient in double,
 *       rounded once to float).
 *   R6  dispatch rows of one expert are in ascending token order; offsets
 *       are the exclusive scan of the per-expert counts.
 *   R7  one 128-wide K slab of a block-scaled GEMM is summed exactly (double)
 *       and rounded once to float; it is promoted with
 *       acc = fmaf(partial, sa * sw, acc), sa * sw a float32 product.
 *   R8  SiLU(x) = x / (1 + exp(-x)) in float32; h = SiLU(G) * U; h is
 *       quantised per 1x128 tile along I before the down projection.
 *   R9  h'_t = u_t + sum_s y_s + sum_k g_k y_k, summed in double, output float.
 *   R10 bias update: with n = T*K selections, expert e is overloaded when
 *       c_e * E > n and underloaded when c_e * E < n (integer compare);
 *       b_e -= gamma or += gamma in float32; equal load leaves b_e unchanged.
 *   R15 input gradient of the layer: the backward GEMMs follow the
 *       forward's FP8 rule (see orc_layer_backward_dgrad).
 *   R16 weight gradients: the FP8 tensors the layer holds are dequantised,
 *       transposed and re-quantised in 128x1 tiles along each expert's
 *       dispatch rows; both operands of the token-contracted GEMM carry a
 *       scale per row per slab (see orc_layer_backward_wgrad).
 *   R14 group-limited routing (the pages: a token goes to at most M = 4
 *       nodes, no scoring rule given): experts form n_groups contiguous
 *       groups; group score = float32 sum, largest first, of the group's
 *       group_topk largest z; keep the topk_groups best groups (equal: lower
 *       group index); then R4 among the kept groups' experts.  Also flagged
 *       as a near tie: the last kept and the next group score differ by
 *       less than 1e-6.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* E4M3 codec (R1)                                                      */
/* ------------------------------------------------------------------ */

/* Decode one E4M3FN code: sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent 0 is subnormal (m * 2^-9); S.1111.111 is NaN; no infinity. */
double orc_e4m3_decode(uint8_t code) {
    int sign = code >> 7;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = m * ldexp(1.0, -9);
    else
        mag = (1.0 + m / 8.0) * ldexp(1.0, e - 7);
    return sign ? -mag : mag;
}

/* Magnitudes of the 127 finite non-negative codes 0x00..0x7E, increasing. */
static double g_mag[127];
static int g_mag_ready = 0;

static void init_mag(void) {
    if (g_mag_ready) return;
    for (int c = 0; c < 127; ++c) g_mag[c] = orc_e4m3_decode((uint8_t)c);
    g_mag_ready = 1;
}

/* Encode: nearest finite magnitude, ties to the even code, saturating. */
uint8_t orc_e4m3_encode(float x) {
    init_mag();
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= g_mag[126]) return sign | 126; /* saturate to 448 */
    /* largest code lo with g_mag[lo] <= a (binary search on the table) */
    int lo = 0, hi = 126;
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (g_mag[mid] <= a) lo = mid; else hi = mid;
    }
    double dlo = a - g_mag[lo], dhi = g_mag[lo + 1] - a;
    int c;
    if (dlo < dhi) c = lo;
    else if (dhi < dlo) c = lo + 1;
    else c = (lo % 2 == 0) ? lo : lo + 1;
    return sign | (uint8_t)c;
}

/* Value of every code, filled once from orc_e4m3_decode (used by the GEMM). */
static double g_dec[256];
static int g_dec_ready = 0;

static void init_dec(void) {
    if (g_dec_ready) return;
    for (int c = 0; c < 256; ++c) g_dec[c] = orc_e4m3_decode((uint8_t)c);
    g_dec_ready = 1;
}

void orc_e4m3_encode_array(const float* x, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(x[i]);
}

static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ------------------------------------------------------------------ */
/* Fine-grained quantisation (R2): [TH] Key ideas FP8; [YLY] §4.3        */
/* ------------------------------------------------------------------ */

/* Quantise n values of one tile with a shared scale. */
static float quant_tile(const float* x, int n, int stride, uint8_t* q, int qstride) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(x[(int64_t)i * stride]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
        for (int i = 0; i < n; ++i) q[(int64_t)i * qstride] = 0x00;
        return 1.0f;
    }
    float scale = amax / 448.0f;
    for (int i = 0; i < n; ++i) {
        float v = x[(int64_t)i * stride] / scale;
        q[(int64_t)i * qstride] = orc_e4m3_encode(v);
    }
    return scale;
}

/* Activations: one scale per 1x128 tile of a row.  x float32 [M, D];
 * q [M, D]; scales [M, D/128] (row-major, oracle's own layout). */
void orc_quant_1x128_f32(const float* x, int M, int D, uint8_t* q, float* scales) {
    int nb = D / 128;
    for (int r = 0; r < M; ++r)
        for (int b = 0; b < nb; ++b)
            scales[(int64_t)r * nb + b] =
                quant_tile(x + (int64_t)r * D + b * 128, 128, 1, q + (int64_t)r * D + b * 128, 1);
}

/* Same for a bfloat16 input (each value widened exactly to float32). */
void orc_quant_1x128_bf16(const uint16_t* x, int M, int D, uint8_t* q, float* scales) {
    float* row = (float*)malloc(sizeof(float) * (size_t)D);
    int nb = D / 128;
    for (int r = 0; r < M; ++r) {
        for (int j = 0; j < D; ++j) row[j] = bf16_to_f32(x[(int64_t)r * D + j]);
        for (int b = 0; b < nb; ++b)
            scales[(int64_t)r * nb + b] =
                quant_tile(row + b * 128, 128, 1, q + (int64_t)r * D + b * 128, 1);
    }
    free(row);
}

/* Weights: one scale per 128x128 block.  w float32 [R, C]; q [R, C];
 * scales [R/128, C/128]. */
void orc_quant_128x128(const float* w, int R, int C, uint8_t* q, float* scales) {
    int rb = R / 128, cb = C / 128;
    float* blk = (float*)malloc(sizeof(float) * 128 * 128);
    uint8_t* qb = (uint8_t*)malloc(128 * 128);
    for (int i = 0; i < rb; ++i)
        for (int j = 0; j < cb; ++j) {
            for (int r = 0; r < 128; ++r)
                for (int c = 0; c < 128; ++c)
                    blk[r * 128 + c] = w[(int64_t)(i * 128 + r) * C + j * 128 + c];
            scales[(int64_t)i * cb + j] = quant_tile(blk, 128 * 128, 1, qb, 1);
            for (int r = 0; r < 128; ++r)
                for (int c = 0; c < 128; ++c)
                    q[(int64_t)(i * 128 + r) * C + j * 128 + c] = qb[r * 128 + c];
        }
    free(blk);
    free(qb);
}

/* ------------------------------------------------------------------ */
/* Block-scaled FP8 GEMM with FP32 promotion every 128 (R7)              */
/* [TH] Key ideas FP8 (N_c = 128); [YLY] §4.3 increased accumulation       */
/* ------------------------------------------------------------------ */

/* out[m, n] = sum over K slabs of (exact slab dot product) * sa * sw,
 * accumulated in float32 with fmaf.
 *   qa [M, Kd] codes, sa [M, Kd/128];  qw [N, Kd] codes, sw [N/128, Kd/128]. */
void orc_gemm_fp8(const uint8_t* qa, const float* sa, int M, int Kd,
                  const uint8_t* qw, const float* sw, int N, float* out) {
    int kb_n = Kd / 128;
    init_dec();
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            float acc = 0.0f;
            for (int kb = 0; kb < kb_n; ++kb) {
                double p = 0.0;
                for (int k = kb * 128; k < kb * 128 + 128; ++k)
                    p += g_dec[qa[(int64_t)m * Kd + k]] * g_dec[qw[(int64_t)n * Kd + k]];
                float s = sa[(int64_t)m * kb_n + kb] * sw[(int64_t)(n / 128) * kb_n + kb];
                acc = fmaf((float)p, s, acc);
            }
            out[(int64_t)m * N + n] = acc;
        }
}

/* Gate/up half of one expert FFN (R7, R8): h = SiLU(A Wg^T) * (A Wu^T),
 * quantised per 1x128 tile along I.
 *   qa [M, d], sa [M, d/128]; wg, wu [I, d] with sg, su [I/128, d/128];
 *   outputs qh [M, I] codes and sh [M, I/128] scales.                      */
void orc_gate_up(const uint8_t* qa, const float* sa, int M, int d, int I,
                 const uint8_t* wg, const float* sg, const uint8_t* wu, const float* su,
                 uint8_t* qh, float* sh) {
    float* G = (float*)malloc(sizeof(float) * (size_t)M * I);
    float* U = (float*)malloc(sizeof(float) * (size_t)M * I);
    orc_gemm_fp8(qa, sa, M, d, wg, sg, I, G);
    orc_gemm_fp8(qa, sa, M, d, wu, su, I, U);
    for (int64_t i = 0; i < (int64_t)M * I; ++i) {
        float g = G[i];
        float silu = g / (1.0f + expf(-g));
        G[i] = silu * U[i]; /* G now holds h */
    }
    orc_quant_1x128_f32(G, M, I, qh, sh);
    free(G); free(U);
}

/* One expert FFN on quantised activation rows: the gate/up half, then the
 * down projection of the quantised h (R7, R8).
 *   wd [d, I] with sd [d/128, I/128]; y [M, d] float32.                    */
void orc_expert_ffn(const uint8_t* qa, const float* sa, int M, int d, int I,
                    const uint8_t* wg, const float* sg, const uint8_t* wu, const float* su,
                    const uint8_t* wd, const float* sd, float* y) {
    uint8_t* qh = (uint8_t*)malloc((size_t)M * I);
    float* sh = (float*)malloc(sizeof(float) * (size_t)M * (I / 128));
    orc_gate_up(qa, sa, M, d, I, wg, sg, wu, su, qh, sh);
    orc_gemm_fp8(qh, sh, M, I, wd, sd, d, y);
    free(qh); free(sh);
}

/* ------------------------------------------------------------------ */
/* Router (R3, R4, R5): [TH] §2 equations for s_{i,t} and g'_{i,t};      */
/* [DB] "Auxiliary-Loss-Free Load Balancing"                             */
/* ------------------------------------------------------------------ */

/* For each token t: s_i = sigmoid(u_t . e_i); top-K of z_i = s_i + b_i;
 * gates = selected s normalised to sum 1.
 *   u bf16 [T, d]; cent [E, d]; bias [E];  outputs idx, gate [T, K],
 *   tie [T] (1 = near tie at the K/K+1 boundary), counts [E] (may be NULL),
 *   scores [T, E] (s values, may be NULL). */
void orc_route(const uint16_t* u, const float* cent, const float* bias,
               int T, int d, int E, int K,
               int32_t* idx, float* gate, uint8_t* tie, int32_t* counts, float* scores) {
    float* s = (float*)malloc(sizeof(float) * (size_t)E);
    float* z = (float*)malloc(sizeof(float) * (size_t)E);
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    if (counts) memset(counts, 0, sizeof(int32_t) * (size_t)E);
    for (int t = 0; t < T; ++t) {
        for (int i = 0; i < E; ++i) {
            double l = 0.0;
            for (int j = 0; j < d; ++j)
                l += (double)bf16_to_f32(u[(int64_t)t * d + j]) * (double)cent[(int64_t)i * d + j];
            float lf = (float)l;
            s[i] = (float)(1.0 / (1.0 + exp(-(double)lf)));
            z[i] = s[i] + bias[i];
            taken[i] = 0;
            if (scores) scores[(int64_t)t * E + i] = s[i];
        }
        /* Selection: K+1 passes of "largest z, lowest index on equality". */
        float zk = 0.0f, zk1 = 0.0f;
        double ssum = 0.0;
        for (int k = 0; k < K + 1 && k < E; ++k) {
            int best = -1;
            for (int i = 0; i < E; ++i) {
                if (taken[i]) continue;
                if (best < 0 || z[i] > z[best]) best = i;
            }
            taken[best] = 1;
            if (k < K) {
                idx[(int64_t)t * K + k] = best;
                ssum += (double)s[best];
                if (k == K - 1) zk = z[best];
                if (counts) counts[best] += 1;
            } else {
                zk1 = z[best];
            }
        }
        for (int k = 0; k < K; ++k)
            gate[(int64_t)t * K + k] = (float)((double)s[idx[(int64_t)t * K + k]] / ssum);
        tie[t] = (K < E && (zk - zk1) < 1e-6f) ? 1 : 0;
    }
    free(s); free(z); free(taken);
}

/* ------------------------------------------------------------------ */
/* Group-limited routing (R14).  The pages: each token is sent to at    */
/* most M = 4 nodes ("官方揭秘DeepSeek-V3模型训练全流程" §2.2 bullet on  */
/* node-limited routing; "DeepSeek V3技術報告", table of innovations).    */
/* Reading: experts form n_groups contiguous groups of E / n_groups      */
/* (one per node); a group's score is the float32 sum, largest first, of */
/* its group_topk largest biased scores z = s + b; the topk_groups groups */
/* with the largest scores are kept (equal scores: lower group index);   */
/* top-K by z among the kept groups' experts as in orc_route; gates as   */
/* in orc_route.  tie: the K-th and (K+1)-th kept z differ by < 1e-6, or */
/* the topk_groups-th and the next group score differ by < 1e-6.         */
/* ------------------------------------------------------------------ */
void orc_route_grouped(const uint16_t* u, const float* cent, const float* bias,
                       int T, int d, int E, int K, int n_groups, int topk_groups,
                       int group_topk, int32_t* idx, float* gate, uint8_t* tie,
                       int32_t* counts, float* scores) {
    const int gsize = E / n_groups;
    float* s = (float*)malloc(sizeof(float) * (size_t)E);
    float* z = (float*)malloc(sizeof(float) * (size_t)E);
    float* gscore = (float*)malloc(sizeof(float) * (size_t)n_groups);
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    unsigned char* kept = (unsigned char*)malloc((size_t)n_groups);
    if (counts) memset(counts, 0, sizeof(int32_t) * (size_t)E);
    for (int t = 0; t < T; ++t) {
        for (int i = 0; i < E; ++i) {
            double l = 0.0;
            for (int j = 0; j < d; ++j)
                l += (double)bf16_to_f32(u[(int64_t)t * d + j]) * (double)cent[(int64_t)i * d + j];
            float lf = (float)l;
            s[i] = (float)(1.0 / (1.0 + exp(-(double)lf)));
            z[i] = s[i] + bias[i];
            if (scores) scores[(int64_t)t * E + i] = s[i];
        }
        /* group scores: group_topk passes of "largest z" inside each group */
        for (int g = 0; g < n_groups; ++g) {
            float acc = 0.0f;
            for (int i = 0; i < E; ++i) taken[i] = 0;
            for (int k = 0; k < group_topk; ++k) {
                int best = -1;
                for (int i = g * gsize; i < (g + 1) * gsize; ++i) {
                    if (taken[i]) continue;
                    if (best < 0 || z[i] > z[best]) best = i;
                }
                taken[best] = 1;
                acc += z[best];
            }
            gscore[g] = acc;
            kept[g] = 0;
        }
        /* kept groups: topk_groups (+1) passes over the group scores */
        float gm = 0.0f, gm1 = 0.0f;
        for (int k = 0; k < topk_groups + 1 && k < n_groups; ++k) {
            int best = -1;
            for (int g = 0; g < n_groups; ++g) {
                if (kept[g] == 1) continue;
                if (best < 0 || gscore[g] > gscore[best]) best = g;
            }
            if (k < topk_groups) {
                kept[best] = 1;
                if (k == topk_groups - 1) gm = gscore[best];
            } else {
                gm1 = gscore[best];
            }
        }
        /* experts of the other groups are out of the selection */
        int allowed = 0;
        for (int i = 0; i < E; ++i) {
            taken[i] = kept[i / gsize] ? 0 : 1;
            allowed += !taken[i];
        }
        float zk = 0.0f, zk1 = 0.0f;
        double ssum = 0.0;
        for (int k = 0; k < K + 1 && k < allowed; ++k) {
            int best = -1;
            for (int i = 0; i < E; ++i) {
                if (taken[i]) continue;
                if (best < 0 || z[i] > z[best]) best = i;
            }
            taken[best] = 1;
            if (k < K) {
                idx[(int64_t)t * K + k] = best;
                ssum += (double)s[best];
                if (k == K - 1) zk = z[best];
                if (counts) counts[best] += 1;
            } else {
                zk1 = z[best];
            }
        }
        for (int k = 0; k < K; ++k)
            gate[(int64_t)t * K + k] = (float)((double)s[idx[(int64_t)t * K + k]] / ssum);
        const int ktie = K < allowed && (zk - zk1) < 1e-6f;
        const int gtie = topk_groups < n_groups && (gm - gm1) < 1e-6f;
        tie[t] = (ktie || gtie) ? 1 : 0;
    }
    free(s); free(z); free(gscore); free(taken); free(kept);
}

/* ------------------------------------------------------------------ */
/* Dispatch (R6): counting sort of (token, slot) pairs by expert.        */
/* [YLY] §2.2: no token is dropped, so every pair gets a row.            */
/* ------------------------------------------------------------------ */

/* counts [E], offsets [E+1], perm_token [T*K] (row -> token),
 * inv_row [T*K] ((t, k) -> row).  Returns 0, or -1 on an expert index
 * outside [0, E). */
int orc_dispatch(const int32_t* idx, int T, int K, int E,
                 int32_t* counts, int32_t* offsets, int32_t* perm_token, int32_t* inv_row) {
    memset(counts, 0, sizeof(int32_t) * (size_t)E);
    for (int64_t p = 0; p < (int64_t)T * K; ++p) {
        if (idx[p] < 0 || idx[p] >= E) return -1;
        counts[idx[p]] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int t = 0; t < T; ++t)           /* ascending token order */
        for (int k = 0; k < K; ++k) {
            int e = idx[(int64_t)t * K + k];
            int row = offsets[e] + fill[e]++;
            perm_token[row] = t;
            inv_row[(int64_t)t * K + k] = row;
        }
    free(fill);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Layer output (R9): [TH] §2 equation for h'_t                          */
/* ------------------------------------------------------------------ */

/* h'_t for the listed tokens.  Expert weights are passed per group:
 * groups 0..E-1 are routed, E..E+S-1 shared; a routed group that no listed
 * token selects may be NULL.  idx, gate [T, K] are the routing of all T
 * tokens (only the listed rows are read).  out [n_tok, d] float32. */
void orc_layer_forward(const uint16_t* u, int T, int d, int E, int K, int S, int I,
                       const int32_t* idx, const float* gate,
                       const uint8_t* const* wg, const float* const* sg,
                       const uint8_t* const* wu, const float* const* su,
                       const uint8_t* const* wd, const float* const* sd,
                       const int32_t* tok, int n_tok, float* out) {
    (void)T; /* idx and gate have T rows; only the listed ones are read */
    uint8_t* qa = (uint8_t*)malloc((size_t)d);
    float* sa = (float*)malloc(sizeof(float) * (size_t)(d / 128));
    float* y = (float*)malloc(sizeof(float) * (size_t)d);
    double* h = (double*)malloc(sizeof(double) * (size_t)d);
    for (int n = 0; n < n_tok; ++n) {
        int t = tok[n];
        const uint16_t* ut = u + (int64_t)t * d;
        /* the quantised activation is the same for every expert (row-local) */
        orc_quant_1x128_bf16(ut, 1, d, qa, sa);
        for (int j = 0; j < d; ++j) h[j] = (double)bf16_to_f32(ut[j]);
        for (int s = 0; s < S; ++s) {
            int g = E + s;
            orc_expert_ffn(qa, sa, 1, d, I, wg[g], sg[g], wu[g], su[g], wd[g], sd[g], y);
            for (int j = 0; j < d; ++j) h[j] += (double)y[j];
        }
        for (int k = 0; k < K; ++k) {
            int g = idx[(int64_t)t * K + k];
            orc_expert_ffn(qa, sa, 1, d, I, wg[g], sg[g], wu[g], su[g], wd[g], sd[g], y);
            double gk = (double)gate[(int64_t)t * K + k];
            for (int j = 0; j < d; ++j) h[j] += gk * (double)y[j];
        }
        for (int j = 0; j < d; ++j) out[(int64_t)n * d + j] = (float)h[j];
    }
    free(qa); free(sa); free(y); free(h);
}

/* ------------------------------------------------------------------ */
/* Input gradient of the layer (R15).  The pages say only that FP8       */
/* carries the inputs and part of the gradient propagation while master  */
/* weights and gradients stay in 16/32 bits ("DeepSeek V3技術報告", FP8   */
/* 資料格式訓練), and ask for transposed-GEMM support in hardware          */
/* ("官方揭秘DeepSeek-V3模型训练全流程", hardware suggestions).  Reading: */
/* every expert backward GEMM follows the forward's FP8 rule -- operand   */
/* rows quantised per 1x128 tile, weights as their 128x128 blocks (W^T    */
/* uses the same codes and block scales, transposed), promotion per 128:  */
/*   dy = g_k dh (routed; float32 product) or dh (shared), quantised;     */
/*   dH = bf16(dy W_down)                    (W_down^T as the B operand); */
/*   G, U recomputed as in the forward; sigma = 1 / (1 + exp(-G));         */
/*   dG = dH U sigma (1 + G (1 - sigma)), dU = dH G sigma (float32);      */
/*   [dG | dU] quantised per 1x128 tile along 2I;                          */
/*   dA = bf16([dG | dU] [W_gate ; W_up])    (contraction over 2I);        */
/*   du = dh + sum_shared dA + sum_routed dA                               */
/*        + sum_k dl_k e_k, with dg_k = dh . y_k (y_k the forward's       */
/*        bf16 expert output), ds_k = (dg_k - sum_j g_j dg_j) / sum_j s_j, */
/*        dl_k = ds_k s_k (1 - s_k)  (the gates' dependence on u through  */
/*        s = sigmoid(u . e); the bias has no gradient).                   */
/* ------------------------------------------------------------------ */

/* float32 -> bfloat16 (round to nearest even) -> float32 */
static float bf16_round(float x) {
    uint32_t b;
    memcpy(&b, &x, 4);
    if ((b & 0x7f800000u) == 0x7f800000u) return x;
    b += 0x7fffu + ((b >> 16) & 1u);
    b &= 0xffff0000u;
    float y;
    memcpy(&y, &b, 4);
    return y;
}

/* W [R, C] codes with block scales [R/128, C/128] -> W^T [C, R], [C/128, R/128] */
static void transpose_blocks(const uint8_t* q, const float* s, int R, int C, uint8_t* qt,
                             float* st) {
    for (int r = 0; r < R; ++r)
        for (int c = 0; c < C; ++c) qt[(int64_t)c * R + r] = q[(int64_t)r * C + c];
    for (int i = 0; i < R / 128; ++i)
        for (int j = 0; j < C / 128; ++j) st[(int64_t)j * (R / 128) + i] = s[(int64_t)i * (C / 128) + j];
}

/* du [n_tok, d] float32 for the listed tokens; dh [T, d] bf16 upstream
 * gradient of h'; idx, gate [T, K] the forward's routing; cent [E, d]. */
void orc_layer_backward_dgrad(const uint16_t* u, int T, int d, int E, int K, int S, int I,
                              const float* cent, const int32_t* idx, const float* gate,
                              const uint8_t* const* wg, const float* const* sg,
                              const uint8_t* const* wu, const float* const* su,
                              const uint8_t* const* wd, const float* const* sd,
                              const uint16_t* dh, const int32_t* tok, int n_tok, float* du) {
    (void)T;
    uint8_t* qa = (uint8_t*)malloc((size_t)d);
    float* sa = (float*)malloc(sizeof(float) * (size_t)(d / 128));
    float* G = (float*)malloc(sizeof(float) * (size_t)I);
    float* U = (float*)malloc(sizeof(float) * (size_t)I);
    float* h = (float*)malloc(sizeof(float) * (size_t)I);
    uint8_t* qh = (uint8_t*)malloc((size_t)I);
    float* sh = (float*)malloc(sizeof(float) * (size_t)(I / 128));
    float* y = (float*)malloc(sizeof(float) * (size_t)d);
    float* dy = (float*)malloc(sizeof(float) * (size_t)d);
    uint8_t* qdy = (uint8_t*)malloc((size_t)d);
    float* sdy = (float*)malloc(sizeof(float) * (size_t)(d / 128));
    float* dH = (float*)malloc(sizeof(float) * (size_t)I);
    float* dgu = (float*)malloc(sizeof(float) * (size_t)2 * I);
    uint8_t* qgu = (uint8_t*)malloc((size_t)2 * I);
    float* sgu = (float*)malloc(sizeof(float) * (size_t)(2 * I / 128));
    float* dA = (float*)malloc(sizeof(float) * (size_t)d);
    float* dhf = (float*)malloc(sizeof(float) * (size_t)d);
    double* acc = (double*)malloc(sizeof(double) * (size_t)d);
    double* dg = (double*)malloc(sizeof(double) * (size_t)K);
    uint8_t* wdT = (uint8_t*)malloc((size_t)I * d);
    float* sdT = (float*)malloc(sizeof(float) * (size_t)(I / 128) * (d / 128));
    uint8_t* wguT = (uint8_t*)malloc((size_t)d * 2 * I);
    float* sguT = (float*)malloc(sizeof(float) * (size_t)(d / 128) * (2 * I / 128));
    uint8_t* tq = (uint8_t*)malloc((size_t)d * I);
    float* ts = (float*)malloc(sizeof(float) * (size_t)(d / 128) * (I / 128));
    const int nI = I / 128, nd = d / 128;
    for (int n = 0; n < n_tok; ++n) {
        const int t = tok[n];
        const uint16_t* ut = u + (int64_t)t * d;
        orc_quant_1x128_bf16(ut, 1, d, qa, sa);
        for (int j = 0; j < d; ++j) {
            dhf[j] = bf16_to_f32(dh[(int64_t)t * d + j]);
            acc[j] = (double)dhf[j];
        }
        for (int q = 0; q < S + K; ++q) {
            const int shared = q < S;
            const int g = shared ? E + q : idx[(int64_t)t * K + (q - S)];
            const float gk = shared ? 1.0f : gate[(int64_t)t * K + (q - S)];
            /* the forward pieces, recomputed */
            orc_gemm_fp8(qa, sa, 1, d, wg[g], sg[g], I, G);
            orc_gemm_fp8(qa, sa, 1, d, wu[g], su[g], I, U);
            for (int i = 0; i < I; ++i) h[i] = G[i] / (1.0f + expf(-G[i])) * U[i];
            orc_quant_1x128_f32(h, 1, I, qh, sh);
            orc_gemm_fp8(qh, sh, 1, I, wd[g], sd[g], d, y);
            /* gradient of the expert output, quantised per 1x128 tile */
            for (int j = 0; j < d; ++j) dy[j] = shared ? dhf[j] : gk * dhf[j];
            orc_quant_1x128_f32(dy, 1, d, qdy, sdy);
            /* dH = dy W_down (B operand W_down^T [I, d]) */
            transpose_blocks(wd[g], sd[g], d, I, wdT, sdT);
            orc_gemm_fp8(qdy, sdy, 1, d, wdT, sdT, I, dH);
            for (int i = 0; i < I; ++i) dH[i] = bf16_round(dH[i]);
            /* SiLU backward */
            for (int i = 0; i < I; ++i) {
                const float sgm = 1.0f / (1.0f + expf(-G[i]));
                dgu[i] = dH[i] * U[i] * sgm * (1.0f + G[i] * (1.0f - sgm));
                dgu[I + i] = dH[i] * G[i] * sgm;
            }
            orc_quant_1x128_f32(dgu, 1, 2 * I, qgu, sgu);
            /* dA = [dG | dU] [W_gate ; W_up]: B operand [W_gate^T | W_up^T] [d, 2I] */
            transpose_blocks(wg[g], sg[g], I, d, tq, ts);
            for (int r = 0; r < d; ++r) memcpy(wguT + (int64_t)r * 2 * I, tq + (int64_t)r * I, (size_t)I);
            for (int i = 0; i < nd; ++i) memcpy(sguT + (int64_t)i * 2 * nI, ts + (int64_t)i * nI, sizeof(float) * nI);
            transpose_blocks(wu[g], su[g], I, d, tq, ts);
            for (int r = 0; r < d; ++r) memcpy(wguT + (int64_t)r * 2 * I + I, tq + (int64_t)r * I, (size_t)I);
            for (int i = 0; i < nd; ++i) memcpy(sguT + (int64_t)i * 2 * nI + nI, ts + (int64_t)i * nI, sizeof(float) * nI);
            orc_gemm_fp8(qgu, sgu, 1, 2 * I, wguT, sguT, d, dA);
            for (int j = 0; j < d; ++j) acc[j] += (double)bf16_round(dA[j]);
            if (!shared) {
                double s_ = 0.0;
                for (int j = 0; j < d; ++j) s_ += (double)dhf[j] * (double)bf16_round(y[j]);
                dg[q - S] = s_;
            }
        }
        /* the gates' dependence on u through s = sigmoid(u . e) */
        double ssum = 0.0, gdg = 0.0;
        double* sk = (double*)malloc(sizeof(double) * (size_t)K);
        for (int k = 0; k < K; ++k) {
            const int e = idx[(int64_t)t * K + k];
            double l = 0.0;
            for (int j = 0; j < d; ++j) l += (double)bf16_to_f32(ut[j]) * (double)cent[(int64_t)e * d + j];
            const float lf = (float)l;
            sk[k] = (double)(float)(1.0 / (1.0 + exp(-(double)lf)));
            ssum += sk[k];
            gdg += (double)gate[(int64_t)t * K + k] * dg[k];
        }
        for (int k = 0; k < K; ++k) {
            const int e = idx[(int64_t)t * K + k];
            const double dl = (dg[k] - gdg) / ssum * sk[k] * (1.0 - sk[k]);
            for (int j = 0; j < d; ++j) acc[j] += dl * (double)cent[(int64_t)e * d + j];
        }
        free(sk);
        for (int j = 0; j < d; ++j) du[(int64_t)n * d + j] = (float)acc[j];
    }
    free(qa); free(sa); free(G); free(U); free(h); free(qh); free(sh); free(y); free(dy);
    free(qdy); free(sdy); free(dH); free(dgu); free(qgu); free(sgu); free(dA); free(dhf);
    free(acc); free(dg); free(wdT); free(sdT); free(wguT); free(sguT); free(tq); free(ts);
}

/* ------------------------------------------------------------------ */
/* Weight gradients of one expert (R16).  The pages keep master weights  */
/* and their gradients in 16/32 bits and FP8 activations in storage      */
/* ("DeepSeek V3技術報告", FP8 資料格式訓練; "官方揭秘DeepSeek-V3模型训练 */
/* 全流程" §4.3 low-precision storage), and ask for transposed GEMMs in   */
/* hardware (same page, hardware suggestions) because the FP8 tensors     */
/* the forward holds in 1x128 tiles along features must be contracted     */
/* over tokens here.  Reading: the four FP8 tensors the layer already     */
/* holds -- the activation rows A and h of the forward, dy and [dG | dU]  */
/* of the input gradient (R15) -- are each dequantised (x = dec(q) s, a   */
/* float32 product), transposed and re-quantised in 128x1 tiles: 128      */
/* consecutive dispatch rows of one expert (the expert's last block       */
/* ragged; a block never spans two experts) by one column, with R2's      */
/* rule.  Then dW_down = dy^T h and [dW_gate ; dW_up] = [dG | dU]^T A,    */
/* each entry summed over 128-row slabs with R7's promotion, where both   */
/* operands carry one scale per row per slab:                            */
/*   acc = fmaf(p, sA * sB, acc),  sA * sB a float32 product.             */
/* Output float32.  An expert that no token selected gets dW = 0.         */
/* ------------------------------------------------------------------ */

/* q [M, C] codes with 1x128 scales s [M, C/128] -> the 128x1 form:
 * qt [C, Mp] codes (Mp = M rounded up to 128; codes past row M are 0) and
 * st [C, Mp/128] scales. */
void orc_requant_128x1(const uint8_t* q, const float* s, int M, int C, uint8_t* qt, float* st) {
    const int nb = (M + 127) / 128, Mp = nb * 128;
    float* col = (float*)malloc(sizeof(float) * 128);
    init_dec();
    for (int c = 0; c < C; ++c)
        for (int b = 0; b < nb; ++b) {
            const int r0 = b * 128, n = M - r0 < 128 ? M - r0 : 128;
            for (int i = 0; i < n; ++i) {
                const float v = (float)g_dec[q[(int64_t)(r0 + i) * C + c]];
                col[i] = v * s[(int64_t)(r0 + i) * (C / 128) + c / 128];
            }
            uint8_t* dst = qt + (int64_t)c * Mp + r0;
            st[(int64_t)c * nb + b] = quant_tile(col, n, 1, dst, 1);
            for (int i = n; i < 128; ++i) dst[i] = 0x00;
        }
    free(col);
}

/* out[n, m] = sum over K slabs of (exact slab dot product) * sa * sb with
 * one scale per row per slab on both sides, accumulated in float32 (R16).
 *   qa [Na, Kd], sa [Na, Kd/128];  qb [Nb, Kd], sb [Nb, Kd/128];  out [Na, Nb]. */
void orc_gemm_fp8_rowscaled(const uint8_t* qa, const float* sa, int Na, int Kd,
                            const uint8_t* qb, const float* sb, int Nb, float* out) {
    int kb_n = Kd / 128;
    init_dec();
    for (int n = 0; n < Na; ++n)
        for (int m = 0; m < Nb; ++m) {
            float acc = 0.0f;
            for (int kb = 0; kb < kb_n; ++kb) {
                double p = 0.0;
                for (int k = kb * 128; k < kb * 128 + 128; ++k)
                    p += g_dec[qa[(int64_t)n * Kd + k]] * g_dec[qb[(int64_t)m * Kd + k]];
                float sc = sa[(int64_t)n * kb_n + kb] * sb[(int64_t)m * kb_n + kb];
                acc = fmaf((float)p, sc, acc);
            }
            out[(int64_t)n * Nb + m] = acc;
        }
}

/* dW_gate, dW_up [I, d] and dW_down [d, I] (float32) of group g: routed
 * expert g < E takes the tokens that selected it, in ascending order (R6),
 * with their gates; shared expert g >= E takes every token with weight 1.
 * wg, wu [I, d] and wd [d, I] are that group's weights with their block
 * scales; u, dh [T, d] bf16; idx, gate [T, K] the forward's routing. */
void orc_layer_backward_wgrad(const uint16_t* u, int T, int d, int E, int K, int I,
                              const int32_t* idx, const float* gate, const uint8_t* wg,
                              const float* sg, const uint8_t* wu, const float* su,
                              const uint8_t* wd, const float* sd, const uint16_t* dh, int g,
                              float* dWg, float* dWu, float* dWd) {
    /* the group's dispatch rows */
    int* tok = (int*)malloc(sizeof(int) * (size_t)(T > 0 ? T : 1));
    float* gk = (float*)malloc(sizeof(float) * (size_t)(T > 0 ? T : 1));
    int m = 0;
    for (int t = 0; t < T; ++t) {
        if (g >= E) {
            tok[m] = t; gk[m] = 1.0f; ++m;
            continue;
        }
        for (int k = 0; k < K; ++k)
            if (idx[(int64_t)t * K + k] == g) {
                tok[m] = t; gk[m] = gate[(int64_t)t * K + k]; ++m;
                break;
            }
    }
    if (m == 0) {
        memset(dWg, 0, sizeof(float) * (size_t)I * d);
        memset(dWu, 0, sizeof(float) * (size_t)I * d);
        memset(dWd, 0, sizeof(float) * (size_t)d * I);
        free(tok); free(gk);
        return;
    }
    const int nb = (m + 127) / 128, Mp = nb * 128;
    uint8_t* qa = (uint8_t*)malloc((size_t)m * d);
    float* sa = (float*)malloc(sizeof(float) * (size_t)m * (d / 128));
    float* G = (float*)malloc(sizeof(float) * (size_t)m * I);
    float* U = (float*)malloc(sizeof(float) * (size_t)m * I);
    float* h = (float*)malloc(sizeof(float) * (size_t)m * I);
    uint8_t* qh = (uint8_t*)malloc((size_t)m * I);
    float* sh = (float*)malloc(sizeof(float) * (size_t)m * (I / 128));
    float* dy = (float*)malloc(sizeof(float) * (size_t)m * d);
    uint8_t* qdy = (uint8_t*)malloc((size_t)m * d);
    float* sdy = (float*)malloc(sizeof(float) * (size_t)m * (d / 128));
    uint8_t* wdT = (uint8_t*)malloc((size_t)I * d);
    float* sdT = (float*)malloc(sizeof(float) * (size_t)(I / 128) * (d / 128));
    float* dH = (float*)malloc(sizeof(float) * (size_t)m * I);
    float* dgu = (float*)malloc(sizeof(float) * (size_t)m * 2 * I);
    uint8_t* qgu = (uint8_t*)malloc((size_t)m * 2 * I);
    float* sgu = (float*)malloc(sizeof(float) * (size_t)m * (2 * I / 128));
    uint8_t* at = (uint8_t*)malloc((size_t)d * Mp);
    float* sat = (float*)malloc(sizeof(float) * (size_t)d * nb);
    uint8_t* ht = (uint8_t*)malloc((size_t)I * Mp);
    float* sht = (float*)malloc(sizeof(float) * (size_t)I * nb);
    uint8_t* dyt = (uint8_t*)malloc((size_t)d * Mp);
    float* sdyt = (float*)malloc(sizeof(float) * (size_t)d * nb);
    uint8_t* gut = (uint8_t*)malloc((size_t)2 * I * Mp);
    float* sgut = (float*)malloc(sizeof(float) * (size_t)2 * I * nb);
    float* dWgu = (float*)malloc(sizeof(float) * (size_t)2 * I * d);

    /* the forward's FP8 activation rows and h */
    for (int r = 0; r < m; ++r)
        orc_quant_1x128_bf16(u + (int64_t)tok[r] * d, 1, d, qa + (int64_t)r * d, sa + (int64_t)r * (d / 128));
    orc_gemm_fp8(qa, sa, m, d, wg, sg, I, G);
    orc_gemm_fp8(qa, sa, m, d, wu, su, I, U);
    for (int64_t i = 0; i < (int64_t)m * I; ++i) h[i] = G[i] / (1.0f + expf(-G[i])) * U[i];
    orc_quant_1x128_f32(h, m, I, qh, sh);
    /* the input gradient's FP8 dy and [dG | dU] (R15) */
    for (int r = 0; r < m; ++r)
        for (int j = 0; j < d; ++j) {
            const float v = bf16_to_f32(dh[(int64_t)tok[r] * d + j]);
            dy[(int64_t)r * d + j] = g >= E ? v : gk[r] * v;
        }
    orc_quant_1x128_f32(dy, m, d, qdy, sdy);
    transpose_blocks(wd, sd, d, I, wdT, sdT);
    orc_gemm_fp8(qdy, sdy, m, d, wdT, sdT, I, dH);
    for (int r = 0; r < m; ++r)
        for (int i = 0; i < I; ++i) {
            const int64_t x = (int64_t)r * I + i;
            const float dHv = bf16_round(dH[x]);
            const float sgm = 1.0f / (1.0f + expf(-G[x]));
            dgu[(int64_t)r * 2 * I + i] = dHv * U[x] * sgm * (1.0f + G[x] * (1.0f - sgm));
            dgu[(int64_t)r * 2 * I + I + i] = dHv * G[x] * sgm;
        }
    orc_quant_1x128_f32(dgu, m, 2 * I, qgu, sgu);
    /* dequantise, transpose, re-quantise in 128x1 tiles */
    orc_requant_128x1(qa, sa, m, d, at, sat);
    orc_requant_128x1(qh, sh, m, I, ht, sht);
    orc_requant_128x1(qdy, sdy, m, d, dyt, sdyt);
    orc_requant_128x1(qgu, sgu, m, 2 * I, gut, sgut);
    /* dW_down = dy^T h;  [dW_gate ; dW_up] = [dG | dU]^T A */
    orc_gemm_fp8_rowscaled(dyt, sdyt, d, Mp, ht, sht, I, dWd);
    orc_gemm_fp8_rowscaled(gut, sgut, 2 * I, Mp, at, sat, d, dWgu);
    memcpy(dWg, dWgu, sizeof(float) * (size_t)I * d);
    memcpy(dWu, dWgu + (int64_t)I * d, sizeof(float) * (size_t)I * d);

    free(tok); free(gk); free(qa); free(sa); free(G); free(U); free(h); free(qh); free(sh);
    free(dy); free(qdy); free(sdy); free(wdT); free(sdT); free(dH); free(dgu); free(qgu);
    free(sgu); free(at); free(sat); free(ht); free(sht); free(dyt); free(sdyt); free(gut);
    free(sgut); free(dWgu);
}

/* ------------------------------------------------------------------ */
/* Bias update (R10): [TH] §2 update rule (gamma = 0.001 there);         */
/* [DB] "Auxiliary-Loss-Free Load Balancing"                             */
/* ------------------------------------------------------------------ */

void orc_update_bias(const int32_t* counts, int E, int T, int K, float gamma, float* bias) {
    int64_t n = (int64_t)T * K;
    for (int e = 0; e < E; ++e) {
        int64_t load = (int64_t)counts[e] * E;
        if (load > n) bias[e] = bias[e] - gamma;
        else if (load < n) bias[e] = bias[e] + gamma;
    }
}
