/*
 * moe_oracle.c -- plain, slow CPU oracle for the forward pass of a Qwen3-style
 * sparse Mixture-of-Experts block.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load or call this library.  It shares
 * no code, header, table or helper with the CUDA library; the two only see the
 * same seeded input bytes.
 *
 * What it computes follows the block's forward method as printed on the
 * cnblogs page "大模型-qwen3 MoE 详细解读" (class Qwen3MoeSparseMoeBlock,
 * __init__ / forward, and the line-by-line commentary that follows it):
 *
 *   logits = x · W_routerᵀ                      (gate = Linear(H, E, bias=False))
 *   p      = softmax(logits) in float          (F.softmax(..., dtype=float))
 *   w, idx = topk(p, K)                        (sorted, largest first)
 *   if norm_topk_prob: w /= Σ_k w
 *   out[t] = Σ_k w_k · MLP_{idx_k}(x_t)        (per-expert loop + index_add_)
 *
 * with MLP_e(x) = down_e( silu(gate_e(x)) ⊙ up_e(x) ) -- the gate_proj /
 * up_proj / down_proj expert of the csdn page "MoE架构深度解析：128专家与8激活的
 * 智能路由" (section "128个专家网络的组织结构与参数分布", parameter table), and the
 * load-balance statistic  aux = n · Σ_i f_i · P_i  of that page's section
 * "负载均衡机制".
 *
 * Readings taken where the pages are silent or ambiguous:
 *  - logits are kept in fp32 (no bf16 rounding) unless ORACLE_BF16_LOGITS;
 *  - ranking uses the fp32 logits, descending, ties to the lower expert index;
 *  - routing weights stay fp32 (no cast to bf16);
 *  - the SwiGLU intermediate a = silu(g)·u is rounded to bf16 (the dtype the
 *    second projection consumes) unless ORACLE_FP64_INTERMEDIATE;
 *  - the token-expert pairs are ordered by expert, then token;
 *  - f_e = counts_e / (T·K) and P_e = mean over tokens of the full softmax.
 *
 * Arithmetic: every dot product and sum is accumulated in double, from the
 * exact values of the bf16 inputs (a bf16×bf16 product is exact in double).
 * Results are rounded once, to fp32 for logits / weights / aux and to bf16
 * (round to nearest even) for the block output.  No blocking, fusion or
 * reordering beyond the definition; OpenMP only splits independent tokens.
 *
 * All arrays are host memory, row-major, contiguous.  bf16 values are passed
 * as their uint16 bit patterns.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BF16_LOGITS 1       /* round logits to bf16 before routing      */
#define ORACLE_FP64_INTERMEDIATE 2 /* keep silu(g)*u in double (no bf16 round) */

/* ---- number formats --------------------------------------------------- */

/* Exact value of a bf16 bit pattern: bf16 is the top half of an IEEE fp32. */
double oracle_bf16_to_f64(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double straight to bf16, to nearest, ties to even (no detour
 * through fp32, which would round twice).  bf16 has 8 significant bits and
 * the fp32 exponent range; subnormals are spaced 2^-133 apart. */
uint16_t oracle_f64_to_bf16(double v) {
    if (isnan(v)) return (uint16_t)0x7FC0;
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    double r;
    if (a == 0.0) {
        r = 0.0;
    } else if (isinf(a)) {
        r = INFINITY;
    } else {
        int ex;
        (void)frexp(a, &ex); /* a = fr·2^ex, fr in [0.5, 1) */
        int ulp_exp = ex - 8;
        if (ulp_exp < -133) ulp_exp = -133;
        double q = ldexp(a, -ulp_exp); /* exact: scaling by a power of two */
        r = ldexp(nearbyint(q), ulp_exp);
        if (r >= ldexp(1.0, 128)) r = INFINITY;
    }
    float f = (float)r; /* exact: r is representable in bf16 */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t b = (uint16_t)(u >> 16);
    if (neg) b |= 0x8000u;
    return b;
}

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* ---- step 1: router logits (gate = Linear(H, E, bias=False)) ------------ */

/* logits[t,e] = Σ_h x[t,h]·W_router[e,h], accumulated in double, rounded to
 * fp32 (or to bf16 then widened, with ORACLE_BF16_LOGITS). */
int oracle_router_logits(const uint16_t* x, int T, int H, const uint16_t* Wr,
                         int E, int flags, float* logits) {
    if (T < 0 || H < 1 || E < 1 || (T > 0 && (!x || !logits)) || !Wr) return 1;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double s = 0.0;
            for (int h = 0; h < H; ++h)
                s += oracle_bf16_to_f64(x[(size_t)t * H + h]) *
                     oracle_bf16_to_f64(Wr[(size_t)e * H + h]);
            float l = (float)s;
            if (flags & ORACLE_BF16_LOGITS) l = (float)oracle_bf16_to_f64(oracle_f64_to_bf16(s));
            logits[(size_t)t * E + e] = l;
        }
    }
    return 0;
}

/* ---- step 2: softmax over all E experts (in double) ---------------------- */

/* probs[t,e] = exp(l_e - max_j l_j) / Σ_j exp(l_j - max_j l_j).  Subtracting
 * the row maximum does not change the result (softmax is shift-invariant). */
int oracle_softmax(const float* logits, int T, int E, double* probs) {
    if (T < 0 || E < 1) return 1;
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (size_t)t * E;
        double m = l[0];
        for (int e = 1; e < E; ++e)
            if (l[e] > m) m = l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += exp((double)l[e] - m);
        for (int e = 0; e < E; ++e) probs[(size_t)t * E + e] = exp((double)l[e] - m) / z;
    }
    return 0;
}

/* ---- steps 3-4: top-k selection and optional renormalisation ------------- */

/* "a before b" in the ranking: larger logit first, equal logits -> lower
 * expert index first.  Float comparison, so -0 == +0. */
static int ranks_before(const float* l, int a, int b) {
    if (l[a] > l[b]) return 1;
    if (l[a] < l[b]) return 0;
    return a < b;
}

/* For each token pick the K experts that come first in the ranking, in
 * ranking order; w_k = p[idx_k], divided by Σ_k p[idx_k] when norm != 0.
 *
 * With bias != NULL: a per-expert routing bias for auxiliary-loss-free load
 * balancing (the DeepSeek scheme named in section "第四阶段：更先进的路由方案：
 * DeepSeek 的突破" of the sshipanoo.com page "项目 17：稀疏性的调度艺术：实现双专家
 * MoE 路由（MoE Router）"), read as entering the selection only: the ranking key
 * of expert e is the fp32 sum l_e + b_e, while the weights stay the
 * probabilities p of the unbiased logits. */
int oracle_route_biased(const float* logits, const float* bias, int T, int E, int K, int norm,
                        int32_t* topk_idx, float* topk_w) {
    if (T < 0 || E < 1 || E > 1024 || K < 1 || K > E) return 1;
    if (T == 0) return 0;
    double* probs = (double*)malloc((size_t)T * E * sizeof(double));
    float* keys = (float*)malloc((size_t)T * E * sizeof(float));
    if (!probs || !keys) {
        free(probs);
        free(keys);
        return 2;
    }
    for (size_t i = 0; i < (size_t)T * E; ++i)
        keys[i] = bias ? (float)(logits[i] + bias[i % (size_t)E]) : logits[i];
    oracle_softmax(logits, T, E, probs);
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        const float* l = keys + (size_t)t * E;
        const double* p = probs + (size_t)t * E;
        char taken[1024];
        int32_t sel[1024];
        memset(taken, 0, (size_t)E);
        for (int k = 0; k < K; ++k) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || ranks_before(l, e, best)) best = e;
            }
            taken[best] = 1;
            sel[k] = best;
        }
        double sum = 0.0;
        for (int k = 0; k < K; ++k) sum += p[sel[k]];
        for (int k = 0; k < K; ++k) {
            topk_idx[(size_t)t * K + k] = sel[k];
            double w = p[sel[k]];
            if (norm) w = w / sum;
            topk_w[(size_t)t * K + k] = (float)w;
        }
    }
    free(probs);
    free(keys);
    return 0;
}

int oracle_route_from_logits(const float* logits, int T, int E, int K, int norm,
                             int32_t* topk_idx, float* topk_w) {
    return oracle_route_biased(logits, NULL, T, E, K, norm, topk_idx, topk_w);
}

/* ---- step 5: dispatch (group the token-expert pairs by expert) ---------- */

/* Pairs (t,k) are numbered in the order (expert, token): for each expert in
 * increasing index, the tokens that chose it in increasing token order.
 *   counts[e]    = number of pairs routed to e
 *   offsets[e]   = Σ_{e'<e} counts[e']   (offsets[E] = T·K)
 *   perm_tok[r]  = token of the pair in row r;  perm_slot[r] = its k-slot
 *   inv[t*K+k]   = row of pair (t,k)
 * Unique, because a token selects each expert at most once. */
/* Expert capacity (section "容量因子设计" of the csdn page "MoE架构深度解析：
 * 128专家与8激活的智能路由": capacity = batch tokens / experts × capacity
 * factor), read for K experts per token as C = ceil(cf·T·K/E) pairs: each
 * expert keeps the first C pairs routed to it, in token order, the way the
 * lpnh.cn page's capacity-aware inference routing fills each expert token by
 * token; keep[t*K+k] = 0 for the others (dropped: they add nothing to the
 * block output).  capacity <= 0 keeps every pair. */
int oracle_keep_mask(const int32_t* topk_idx, int T, int E, int K, int capacity, uint8_t* keep) {
    if (T < 0 || E < 1 || K < 1) return 1;
    int32_t* seen = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    if (!seen) return 2;
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            const int e = topk_idx[(size_t)t * K + k];
            if (e < 0 || e >= E) {
                free(seen);
                return 3;
            }
            keep[(size_t)t * K + k] = (uint8_t)(capacity <= 0 || seen[e] < capacity);
            seen[e] += 1;
        }
    free(seen);
    return 0;
}

/* With a capacity, the rows hold the kept pairs only (same order), counts[e]
 * stays the number of pairs routed to e, offsets are prefix sums of the kept
 * counts (offsets[E] = kept pairs) and inv = -1 for a dropped pair. */
int oracle_dispatch_cap(const int32_t* topk_idx, int T, int E, int K, int capacity,
                        int32_t* counts, int32_t* offsets, int32_t* perm_tok, int32_t* perm_slot,
                        int32_t* inv) {
    if (T < 0 || E < 1 || K < 1) return 1;
    uint8_t* keep = (uint8_t*)malloc((size_t)T * K + 1);
    if (!keep) return 2;
    int rc = oracle_keep_mask(topk_idx, T, E, K, capacity, keep);
    if (rc) {
        free(keep);
        return rc;
    }
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (size_t i = 0; i < (size_t)T * K; ++i) counts[topk_idx[i]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        const int kept = capacity > 0 && counts[e] > capacity ? capacity : counts[e];
        offsets[e + 1] = offsets[e] + kept;
    }
    int32_t row = 0;
    for (int e = 0; e < E; ++e)
        for (int t = 0; t < T; ++t)
            for (int k = 0; k < K; ++k)
                if (topk_idx[(size_t)t * K + k] == e) {
                    if (!keep[(size_t)t * K + k]) {
                        inv[(size_t)t * K + k] = -1;
                        continue;
                    }
                    perm_tok[row] = t;
                    perm_slot[row] = k;
                    inv[(size_t)t * K + k] = row;
                    ++row;
                }
    free(keep);
    return 0;
}

int oracle_dispatch(const int32_t* topk_idx, int T, int E, int K, int32_t* counts,
                    int32_t* offsets, int32_t* perm_tok, int32_t* perm_slot, int32_t* inv) {
    return oracle_dispatch_cap(topk_idx, T, E, K, 0, counts, offsets, perm_tok, perm_slot, inv);
}

/* ---- step 6: one expert's SwiGLU MLP on one token ----------------------- */

/* y[h] = Σ_i a_i · W_down[e,h,i],  a_i = silu(g_i)·u_i,
 * g_i = Σ_h x_h·W_gate[e,i,h],  u_i = Σ_h x_h·W_up[e,i,h].
 * Wg/Wu point at expert e's [I,H] block, Wd at its [H,I] block. */
int oracle_expert_mlp(const uint16_t* x_row, int H, const uint16_t* Wg, const uint16_t* Wu,
                      const uint16_t* Wd, int I, int flags, double* y) {
    double* a = (double*)malloc((size_t)I * sizeof(double));
    if (!a) return 2;
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) {
            double xv = oracle_bf16_to_f64(x_row[h]);
            g += xv * oracle_bf16_to_f64(Wg[(size_t)i * H + h]);
            u += xv * oracle_bf16_to_f64(Wu[(size_t)i * H + h]);
        }
        double ai = silu(g) * u;
        if (!(flags & ORACLE_FP64_INTERMEDIATE)) ai = oracle_bf16_to_f64(oracle_f64_to_bf16(ai));
        a[i] = ai;
    }
    for (int h = 0; h < H; ++h) {
        double s = 0.0;
        for (int i = 0; i < I; ++i) s += a[i] * oracle_bf16_to_f64(Wd[(size_t)h * I + i]);
        y[h] = s;
    }
    free(a);
    return 0;
}

/* ---- step 7: combine (weighted sum over the token's K experts) ---------- */

/* out_row[h] = bf16( Σ_k w_k · MLP_{idx_k}(x_row)[h] ), the sum in double.
 * out_f64_row (may be NULL) receives the sum before that final rounding. */
int oracle_token_output_ex(const uint16_t* x_row, int H, const int32_t* idx_row,
                           const float* w_row, int K, const uint16_t* Wg, const uint16_t* Wu,
                           const uint16_t* Wd, int E, int I, int flags, uint16_t* out_row,
                           double* out_f64_row) {
    double* acc = (double*)calloc((size_t)H, sizeof(double));
    double* y = (double*)malloc((size_t)H * sizeof(double));
    if (!acc || !y) { free(acc); free(y); return 2; }
    int rc = 0;
    for (int k = 0; k < K && rc == 0; ++k) {
        int e = idx_row[k];
        if (e < 0 || e >= E) { rc = 3; break; }
        size_t blk = (size_t)I * H;
        rc = oracle_expert_mlp(x_row, H, Wg + (size_t)e * blk, Wu + (size_t)e * blk,
                               Wd + (size_t)e * blk, I, flags, y);
        for (int h = 0; h < H; ++h) acc[h] += (double)w_row[k] * y[h];
    }
    for (int h = 0; h < H; ++h) {
        if (out_row) out_row[h] = oracle_f64_to_bf16(acc[h]);
        if (out_f64_row) out_f64_row[h] = acc[h];
    }
    free(acc);
    free(y);
    return rc;
}

int oracle_token_output(const uint16_t* x_row, int H, const int32_t* idx_row,
                        const float* w_row, int K, const uint16_t* Wg, const uint16_t* Wu,
                        const uint16_t* Wd, int E, int I, int flags, uint16_t* out_row) {
    return oracle_token_output_ex(x_row, H, idx_row, w_row, K, Wg, Wu, Wd, E, I, flags, out_row,
                                  NULL);
}

/* ---- step 8: load-balance statistic ------------------------------------- */

/* aux = E · Σ_e f_e · P_e  with  f_e = counts_e / (T·K)  (share of the
 * token-expert pairs sent to e) and  P_e = (1/T) Σ_t p[t,e]  (mean router
 * probability of e).  T = 0 gives 0. */
double oracle_aux(const double* probs, const int32_t* counts, int T, int E, int K) {
    if (T <= 0) return 0.0;
    double s = 0.0;
    for (int e = 0; e < E; ++e) {
        double P = 0.0;
        for (int t = 0; t < T; ++t) P += probs[(size_t)t * E + e];
        P /= (double)T;
        double f = (double)counts[e] / ((double)T * (double)K);
        s += f * P;
    }
    return (double)E * s;
}

/* ---- the whole block ---------------------------------------------------- */

/* Full forward.  Routing, dispatch and aux cover all T tokens; the block
 * output is produced for the n_rows tokens listed in rows (all tokens, in
 * order, when rows == NULL), into out[n_rows, H] (bf16) and, when out_f64 is
 * not NULL, out_f64[n_rows, H] (the same values before the bf16 rounding).
 * Any of logits / idx / w / aux / counts may be NULL.  Returns 0 on success. */
/* The expert weights of a forward and the step that turns a token's kept
 * pairs into its output row: bf16 matrices (oracle_token_output_ex) or 4-bit
 * groups (token_output_q4 below). */
typedef struct {
    const uint16_t *Wg, *Wu, *Wd;                      /* bf16 [E,I,H], [E,I,H], [E,H,I] */
    const uint8_t *qg, *qu, *qd;                       /* or 4-bit codes of the same shape */
    const uint16_t *sg, *bg, *su, *bu, *sd, *bd;       /* and their group scales / biases */
} experts_t;

static int token_output_q4(const uint16_t* x_row, int H, const int32_t* idx_row,
                           const float* w_row, int K, const experts_t* W, int E, int I,
                           int flags, uint16_t* out_row, double* out_f64_row);

static int experts_token_output(const experts_t* W, const uint16_t* x_row, int H,
                                const int32_t* ik, const float* wk, int nk, int E, int I,
                                int flags, uint16_t* out_row, double* out_f64_row) {
    if (W->qg)
        return token_output_q4(x_row, H, ik, wk, nk, W, E, I, flags, out_row, out_f64_row);
    return oracle_token_output_ex(x_row, H, ik, wk, nk, W->Wg, W->Wu, W->Wd, E, I, flags,
                                  out_row, out_f64_row);
}

static int moe_forward_any(const uint16_t* x, int T, int H, const uint16_t* Wr, const float* bias,
                           int capacity, const experts_t* W, int E, int K, int I, int norm,
                           int flags, const int32_t* rows, int n_rows, uint16_t* out,
                           double* out_f64, float* logits_out, int32_t* idx_out, float* w_out,
                           float* aux_out, int32_t* counts_out) {
    if (T < 0 || H < 1 || E < 1 || E > 1024 || K < 1 || K > E || I < 1) return 1;
    if (T == 0) {
        if (aux_out) *aux_out = 0.0f;
        if (counts_out) for (int e = 0; e < E; ++e) counts_out[e] = 0;
        return 0;
    }
    size_t TE = (size_t)T * E, TK = (size_t)T * K;
    float* logits = (float*)malloc(TE * sizeof(float));
    double* probs = (double*)malloc(TE * sizeof(double));
    int32_t* idx = (int32_t*)malloc(TK * sizeof(int32_t));
    float* w = (float*)malloc(TK * sizeof(float));
    int32_t* counts = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    uint8_t* keep = (uint8_t*)malloc(TK);
    int rc = 0;
    if (!logits || !probs || !idx || !w || !counts || !keep) rc = 2;
    if (!rc) rc = oracle_router_logits(x, T, H, Wr, E, flags, logits);
    if (!rc) rc = oracle_softmax(logits, T, E, probs);
    if (!rc) rc = oracle_route_biased(logits, bias, T, E, K, norm, idx, w);
    if (!rc) {
        for (size_t i = 0; i < TK; ++i) counts[idx[i]] += 1;
        if (aux_out) *aux_out = (float)oracle_aux(probs, counts, T, E, K);
        rc = oracle_keep_mask(idx, T, E, K, capacity, keep);
    }
    if (!rc && (out || out_f64)) {
        int n = rows ? n_rows : T;
        int fail = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
        for (int j = 0; j < n; ++j) {
            int t = rows ? rows[j] : j;
            if (t < 0 || t >= T) { fail |= 1; continue; }
            int32_t ik[1024];  /* the token's kept pairs, in k order */
            float wk[1024];
            int nk = 0;
            for (int k = 0; k < K; ++k)
                if (keep[(size_t)t * K + k]) {
                    ik[nk] = idx[(size_t)t * K + k];
                    wk[nk] = w[(size_t)t * K + k];
                    ++nk;
                }
            if (experts_token_output(W, x + (size_t)t * H, H, ik, wk, nk, E, I, flags,
                                     out ? out + (size_t)j * H : NULL,
                                     out_f64 ? out_f64 + (size_t)j * H : NULL))
                fail |= 1;
        }
        if (fail) rc = 3;
    }
    if (!rc) {
        if (logits_out) memcpy(logits_out, logits, TE * sizeof(float));
        if (idx_out) memcpy(idx_out, idx, TK * sizeof(int32_t));
        if (w_out) memcpy(w_out, w, TK * sizeof(float));
        if (counts_out) memcpy(counts_out, counts, (size_t)E * sizeof(int32_t));
    }
    free(logits);
    free(probs);
    free(idx);
    free(w);
    free(counts);
    free(keep);
    return rc;
}

int oracle_moe_forward_b(const uint16_t* x, int T, int H, const uint16_t* Wr, const float* bias,
                         int capacity, const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd,
                         int E, int K, int I, int norm, int flags, const int32_t* rows, int n_rows,
                         uint16_t* out, double* out_f64, float* logits_out, int32_t* idx_out,
                         float* w_out, float* aux_out, int32_t* counts_out) {
    experts_t W;
    memset(&W, 0, sizeof W);
    W.Wg = Wg;
    W.Wu = Wu;
    W.Wd = Wd;
    return moe_forward_any(x, T, H, Wr, bias, capacity, &W, E, K, I, norm, flags, rows, n_rows,
                           out, out_f64, logits_out, idx_out, w_out, aux_out, counts_out);
}

/* The block forward without a selection bias or a capacity. */
int oracle_moe_forward(const uint16_t* x, int T, int H, const uint16_t* Wr, const uint16_t* Wg,
                       const uint16_t* Wu, const uint16_t* Wd, int E, int K, int I, int norm,
                       int flags, const int32_t* rows, int n_rows, uint16_t* out,
                       double* out_f64, float* logits_out, int32_t* idx_out, float* w_out,
                       float* aux_out, int32_t* counts_out) {
    return oracle_moe_forward_b(x, T, H, Wr, NULL, 0, Wg, Wu, Wd, E, K, I, norm, flags, rows, n_rows,
                                out, out_f64, logits_out, idx_out, w_out, aux_out, counts_out);
}

/* ---- 4-bit group quantisation of the expert weights ----------------------
 *
 * The csdn page "MoE架构深度解析：128专家与8激活的智能路由", section
 * "参数量化与存储优化": the experts' weights are stored as 4-bit values in
 * groups of 128 parameters, each group with its own scale and bias.  The page
 * gives no formula; the reading taken here:
 *   - a group is 128 consecutive entries of one weight row, i.e. along the
 *     projection's input dimension (H for gate_proj / up_proj, I for
 *     down_proj);
 *   - lo, hi = the group's minimum and maximum (a zero minimum taken as +0);
 *     the scale s = bf16(fp32(hi - lo) / 15) and the bias b = lo (a bf16 value
 *     already);
 *   - the code of w is q = clamp(rint(fp32(w - b) / s), 0, 15), every step in
 *     fp32 arithmetic (q = 0 when s = 0);
 *   - the dequantised weight is w' = bf16(q·s + b), rounded once from the
 *     exact value (oracle_dequantize_q4; oracle_dequantize_q4_f64 gives the
 *     exact value itself).
 * A forward with quantised experts is the forward with the weights W'
 * (oracle_moe_forward_q4 computes it from the codes, scales and biases).
 */

static float q4_f32(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* W [rows, cols] bf16 (cols % 128 == 0) -> q [rows, cols] codes 0..15,
 * s, b [rows, cols / 128] bf16. */
int oracle_quantize_q4(const uint16_t* W, int rows, int cols, uint8_t* q, uint16_t* s,
                       uint16_t* b) {
    if (rows < 0 || cols <= 0 || cols % 128) return 1;
    const int groups = cols / 128;
    for (long long r = 0; r < rows; ++r) {
        for (int g = 0; g < groups; ++g) {
            const uint16_t* w = W + r * cols + (long long)g * 128;
            float lo = q4_f32(w[0]), hi = lo;
            for (int j = 1; j < 128; ++j) {
                const float v = q4_f32(w[j]);
                if (v < lo) lo = v;
                if (v > hi) hi = v;
            }
            if (lo == 0.0f) lo = 0.0f; /* a zero minimum is stored as +0 */
            const float span = hi - lo;
            const uint16_t sb = oracle_f64_to_bf16((double)(span / 15.0f));
            const uint16_t bb = oracle_f64_to_bf16((double)lo);
            const float sf = q4_f32(sb), bf = q4_f32(bb);
            for (int j = 0; j < 128; ++j) {
                int code = 0;
                if (sf != 0.0f) {
                    const float t = rintf((q4_f32(w[j]) - bf) / sf);
                    code = t < 0.0f ? 0 : (t > 15.0f ? 15 : (int)t);
                }
                q[r * cols + (long long)g * 128 + j] = (uint8_t)code;
            }
            s[r * groups + g] = sb;
            b[r * groups + g] = bb;
        }
    }
    return 0;
}

/* q, s, b as above -> W' [rows, cols] bf16: w' = bf16(q·s + b).  q·s is exact
 * in double (a 4-bit integer times a bf16); the sum is exact there too unless
 * the two terms lie more than 2^41 apart, and then the sum rounds to b in bf16
 * either way. */
int oracle_dequantize_q4(const uint8_t* q, const uint16_t* s, const uint16_t* b, int rows,
                         int cols, uint16_t* W) {
    if (rows < 0 || cols <= 0 || cols % 128) return 1;
    const int groups = cols / 128;
    for (long long r = 0; r < rows; ++r)
        for (int c = 0; c < cols; ++c) {
            const long long gi = r * groups + c / 128;
            const uint8_t code = q[r * cols + c];
            if (code > 15) return 2;
            const double v = (double)code * oracle_bf16_to_f64(s[gi]) + oracle_bf16_to_f64(b[gi]);
            W[r * cols + c] = oracle_f64_to_bf16(v);
        }
    return 0;
}

/* q, s, b as above -> W [rows, cols] in double: w = q·s + b, exact (q·s is a
 * 4-bit integer times a bf16, exact in double; the sum is exact unless the two
 * terms lie more than 2^44 apart). */
int oracle_dequantize_q4_f64(const uint8_t* q, const uint16_t* s, const uint16_t* b, int rows,
                             int cols, double* W) {
    if (rows < 0 || cols <= 0 || cols % 128) return 1;
    const int groups = cols / 128;
    for (long long r = 0; r < rows; ++r)
        for (int c = 0; c < cols; ++c) {
            const long long g = r * groups + c / 128;
            const uint8_t code = q[r * cols + c];
            if (code > 15) return 2;
            W[r * cols + c] = (double)code * oracle_bf16_to_f64(s[g]) + oracle_bf16_to_f64(b[g]);
        }
    return 0;
}

/* Row `row` of a 4-bit matrix with `cols` columns, as the dequantised
 * weights w' = bf16(q·s + b). */
static void q4_row(const uint8_t* q, const uint16_t* s, const uint16_t* b, size_t row, int cols,
                   double* out) {
    const int groups = cols / 128;
    for (int c = 0; c < cols; ++c) {
        const size_t g = row * (size_t)groups + (size_t)(c / 128);
        const double v = (double)q[row * (size_t)cols + c] * oracle_bf16_to_f64(s[g]) +
                         oracle_bf16_to_f64(b[g]);
        out[c] = oracle_bf16_to_f64(oracle_f64_to_bf16(v));
    }
}

/* oracle_expert_mlp of expert e on 4-bit weights (the dequantised w'). */
static int expert_mlp_q4(const uint16_t* x_row, int H, const experts_t* W, int e, int I,
                         int flags, double* y) {
    double* a = (double*)malloc((size_t)I * sizeof(double));
    double* xr = (double*)malloc((size_t)H * sizeof(double));
    double* wg = (double*)malloc((size_t)H * sizeof(double));
    double* wu = (double*)malloc((size_t)H * sizeof(double));
    double* wd = (double*)malloc((size_t)I * sizeof(double));
    int rc = (a && xr && wg && wu && wd) ? 0 : 2;
    if (!rc) {
        for (int h = 0; h < H; ++h) xr[h] = oracle_bf16_to_f64(x_row[h]);
        for (int i = 0; i < I; ++i) {
            const size_t row = (size_t)e * I + i;
            q4_row(W->qg, W->sg, W->bg, row, H, wg);
            q4_row(W->qu, W->su, W->bu, row, H, wu);
            double g = 0.0, u = 0.0;
            for (int h = 0; h < H; ++h) {
                g += xr[h] * wg[h];
                u += xr[h] * wu[h];
            }
            double ai = silu(g) * u;
            if (!(flags & ORACLE_FP64_INTERMEDIATE)) ai = oracle_bf16_to_f64(oracle_f64_to_bf16(ai));
            a[i] = ai;
        }
        for (int h = 0; h < H; ++h) {
            q4_row(W->qd, W->sd, W->bd, (size_t)e * H + h, I, wd);
            double acc = 0.0;
            for (int i = 0; i < I; ++i) acc += a[i] * wd[i];
            y[h] = acc;
        }
    }
    free(a);
    free(xr);
    free(wg);
    free(wu);
    free(wd);
    return rc;
}

/* oracle_token_output_ex on 4-bit weights. */
static int token_output_q4(const uint16_t* x_row, int H, const int32_t* idx_row,
                           const float* w_row, int K, const experts_t* W, int E, int I,
                           int flags, uint16_t* out_row, double* out_f64_row) {
    double* acc = (double*)calloc((size_t)H, sizeof(double));
    double* y = (double*)malloc((size_t)H * sizeof(double));
    if (!acc || !y) { free(acc); free(y); return 2; }
    int rc = 0;
    for (int k = 0; k < K && rc == 0; ++k) {
        const int e = idx_row[k];
        if (e < 0 || e >= E) { rc = 3; break; }
        rc = expert_mlp_q4(x_row, H, W, e, I, flags, y);
        for (int h = 0; h < H; ++h) acc[h] += (double)w_row[k] * y[h];
    }
    for (int h = 0; h < H; ++h) {
        if (out_row) out_row[h] = oracle_f64_to_bf16(acc[h]);
        if (out_f64_row) out_f64_row[h] = acc[h];
    }
    free(acc);
    free(y);
    return rc;
}

/* The block forward on 4-bit experts: codes q* [E,I,H] / [E,I,H] / [E,H,I]
 * (one byte per code), scales s* and biases b* [E, rows, cols / 128] bf16, as
 * oracle_quantize_q4 writes them; the weights are w' = bf16(q·s + b); every
 * other argument as for oracle_moe_forward_b. */
int oracle_moe_forward_q4(const uint16_t* x, int T, int H, const uint16_t* Wr, const float* bias,
                          int capacity, const uint8_t* qg, const uint16_t* sg, const uint16_t* bg,
                          const uint8_t* qu, const uint16_t* su, const uint16_t* bu,
                          const uint8_t* qd, const uint16_t* sd, const uint16_t* bd, int E, int K,
                          int I, int norm, int flags, const int32_t* rows, int n_rows,
                          uint16_t* out, double* out_f64, float* logits_out, int32_t* idx_out,
                          float* w_out, float* aux_out, int32_t* counts_out) {
    if (H % 128 || I % 128) return 1;
    experts_t W;
    memset(&W, 0, sizeof W);
    W.qg = qg; W.sg = sg; W.bg = bg;
    W.qu = qu; W.su = su; W.bu = bu;
    W.qd = qd; W.sd = sd; W.bd = bd;
    return moe_forward_any(x, T, H, Wr, bias, capacity, &W, E, K, I, norm, flags, rows, n_rows,
                           out, out_f64, logits_out, idx_out, w_out, aux_out, counts_out);
}

/* One token's output on 4-bit experts (oracle_token_output_ex's contract). */
int oracle_token_output_q4(const uint16_t* x_row, int H, const int32_t* idx_row,
                           const float* w_row, int K, const uint8_t* qg, const uint16_t* sg,
                           const uint16_t* bg, const uint8_t* qu, const uint16_t* su,
                           const uint16_t* bu, const uint8_t* qd, const uint16_t* sd,
                           const uint16_t* bd, int E, int I, int flags, uint16_t* out_row,
                           double* out_f64_row) {
    experts_t W;
    memset(&W, 0, sizeof W);
    W.qg = qg; W.sg = sg; W.bg = bg;
    W.qu = qu; W.su = su; W.bu = bu;
    W.qd = qd; W.sd = sd; W.bd = bd;
    return token_output_q4(x_row, H, idx_row, w_row, K, &W, E, I, flags, out_row, out_f64_row);
}
