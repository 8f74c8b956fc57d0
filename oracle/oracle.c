/*
 * oracle.c -- plain, single-threaded CPU restatement of the MoE routing path.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load or call this file. The CUDA library
 * never links, loads or calls it, and the two share no code: no headers, no
 * helpers, no tables. This file is written from the definitions on the pages:
 *
 *   [TE]   NVIDIA TransformerEngine PR 3012, "[Common] Optimize fused router
 *          forward/backward kernels": fused_topk_with_score_function and
 *          fused_score_for_moe_aux_loss, forward and backward; the launcher's
 *          host checks ("Hardening"); the flowchart (score fn, then top-k, then
 *          write probs + routing_map); the byte rule ("Performance").
 *   [FLY]  ROCm FlyDSL PR 582, "Fuse TopKGatingSoftmax and MoE Sorting kernels":
 *          the sorting step that buckets (token, slot) pairs by expert.
 *   [GEMM] ROCm FlyDSL PR 947, "Port moe_gemm_2stage ...": the consumer of the
 *          sorted layout; a sorted id decodes to (token, slot) through a rank-3
 *          [tokens, topk, inter] view, i.e. id = token*topk + slot, and sentinel
 *          rows past the last valid row contribute 0.
 *
 * Where the pages are silent the plainest reading is taken; each reading is
 * marked READING below.
 *
 * Precision. Every value the path outputs is computed here in double. Where
 * floating point decides an integer -- which experts are selected -- the
 * decision is taken in fp32, the kernels' precision, on keys whose fp32
 * arithmetic is fully specified (IEEE add/mul/div/fma, round to nearest even,
 * no contraction: build with -ffp-contract=off, no fast-math):
 *   softmax: key = the logit itself (softmax is strictly increasing in the
 *            logit, so the top-k set of the scores is the top-k set of the
 *            logits; READING);
 *   sigmoid: key = fp32 sigmoid(x) (+ fp32 bias[e] when a bias is given),
 *            with sigmoid computed through orc_expf below.
 * Ties between equal keys go to the lower expert index.
 *
 * Error convention: functions return 0 on success and -1 when an argument
 * violates the stated preconditions; nothing is written in that case.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_SOFTMAX 0
#define ORC_SIGMOID 1

/* ------------------------------------------------------------------------- */
/* fp32 exponential: the written specification both sides implement.         */
/* ------------------------------------------------------------------------- */
/*
 * Method: Cody & Waite argument reduction ("Software Manual for the Elementary
 * Functions", 1980) followed by the degree-7 Taylor polynomial of exp about 0.
 *
 *   n = rint(x * log2(e))                 (fp32 multiply, round half to even)
 *   r = (x - n*LN2_HI) - n*LN2_LO         (two fp32 fma's)
 *   p = sum_{i=0..7} r^i / i!             (Horner, fp32 fma's)
 *   exp(x) = (p * 2^floor_div(n)) * 2^(n - floor_div(n))   (two fp32 multiplies)
 *
 * LN2_HI is ln 2 truncated to 16 fraction bits (15 significant bits), so
 * n*LN2_HI is exact for |n| <= 2^9; LN2_LO = fp32(ln 2 - LN2_HI).
 * With |r| <= ln2/2 the Taylor remainder is below r^8/8! < 5.2e-9 (under 0.1
 * ulp of p), so the total error is a little over 1 ulp. The scale 2^n is
 * applied as two factors, each a normal power of two, so results that fall in
 * the subnormal range round once, in the last multiply. x >= 89 gives +inf and
 * x <= -104 gives +0 (exp(-104) is below half the smallest subnormal).
 */
static const double ORC_LN2 = 0.693147180559945309417232121458176568;

static float orc_ln2_hi(void) { return (float)(floor(ORC_LN2 * 65536.0) / 65536.0); }
static float orc_ln2_lo(void) { return (float)(ORC_LN2 - (double)orc_ln2_hi()); }

static float orc_pow2i(int k) /* 2^k for -126 <= k <= 127 */
{
    uint32_t bits = (uint32_t)(k + 127) << 23;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

float orc_expf(float x)
{
    if (x != x) return x;
    if (x >= 89.0f) return INFINITY;
    if (x <= -104.0f) return 0.0f;
    const float log2e = (float)(1.0 / ORC_LN2);
    const float ln2_hi = orc_ln2_hi();
    const float ln2_lo = orc_ln2_lo();
    /* 1/i! for i = 0..7 */
    const float c0 = 1.0f, c1 = 1.0f, c2 = (float)(1.0 / 2.0), c3 = (float)(1.0 / 6.0),
                c4 = (float)(1.0 / 24.0), c5 = (float)(1.0 / 120.0), c6 = (float)(1.0 / 720.0),
                c7 = (float)(1.0 / 5040.0);
    float t = x * log2e;
    float nf = rintf(t);
    int n = (int)nf;
    float r = fmaf(-nf, ln2_hi, x);
    r = fmaf(-nf, ln2_lo, r);
    float p = c7;
    p = fmaf(p, r, c6);
    p = fmaf(p, r, c5);
    p = fmaf(p, r, c4);
    p = fmaf(p, r, c3);
    p = fmaf(p, r, c2);
    p = fmaf(p, r, c1);
    p = fmaf(p, r, c0);
    int n1 = n / 2; /* C division truncates toward zero */
    int n2 = n - n1;
    float y = p * orc_pow2i(n1);
    y = y * orc_pow2i(n2);
    return y;
}

/* fp32 logistic function used for sigmoid selection keys: 1 / (1 + exp(-x)). */
float orc_sigmoidf(float x)
{
    float e = orc_expf(-x);
    float d = 1.0f + e;
    return 1.0f / d;
}

/* Elementwise forms over arrays, for sweeps. */
void orc_expf_array(const float* x, float* y, size_t n)
{
    for (size_t i = 0; i < n; ++i) y[i] = orc_expf(x[i]);
}

void orc_sigmoidf_array(const float* x, float* y, size_t n)
{
    for (size_t i = 0; i < n; ++i) y[i] = orc_sigmoidf(x[i]);
}

/* ------------------------------------------------------------------------- */
/* Selection order: larger key first; equal keys, lower index first.          */
/* ------------------------------------------------------------------------- */
typedef struct {
    float key;
    int32_t idx;
} orc_kv;

static int orc_kv_cmp(const void* a, const void* b)
{
    const orc_kv* p = (const orc_kv*)a;
    const orc_kv* q = (const orc_kv*)b;
    if (p->key > q->key) return -1;
    if (p->key < q->key) return 1;
    return (p->idx < q->idx) ? -1 : (p->idx > q->idx ? 1 : 0);
}

/* Sort kv[0..n) into selection order. */
static void orc_order(orc_kv* kv, int n) { qsort(kv, (size_t)n, sizeof(orc_kv), orc_kv_cmp); }

/* ------------------------------------------------------------------------- */
/* Scores in double: the score function of [TE] (softmax over all E, or the  */
/* elementwise sigmoid).                                                     */
/* ------------------------------------------------------------------------- */
static void orc_scores(int score_fn, const float* x, int E, double* s)
{
    if (score_fn == ORC_SOFTMAX) {
        double m = (double)x[0];
        for (int e = 1; e < E; ++e)
            if ((double)x[e] > m) m = (double)x[e];
        double den = 0.0;
        for (int e = 0; e < E; ++e) den += exp((double)x[e] - m);
        for (int e = 0; e < E; ++e) s[e] = exp((double)x[e] - m) / den;
    } else {
        for (int e = 0; e < E; ++e) s[e] = 1.0 / (1.0 + exp(-(double)x[e]));
    }
}

/* fp32 selection keys (see the header comment). */
static void orc_keys(int score_fn, const float* x, const float* bias, int E, float* key)
{
    for (int e = 0; e < E; ++e) {
        if (score_fn == ORC_SOFTMAX) {
            key[e] = x[e];
        } else {
            float s = orc_sigmoidf(x[e]);
            key[e] = bias ? s + bias[e] : s;
        }
    }
}

/*
 * Top-k_r selection for one token, optionally group-limited.
 *
 * Group-limited selection (READING of [TE] "group_topk" with the host check
 * "topk % group_topk == 0"): the E experts form n_group contiguous groups of
 * E/n_group; a group's score is the fp32 sum of its m = k_r/topk_group largest
 * keys, added largest first; the topk_group best groups are kept (ties: lower
 * group index) and the k_r experts are chosen among the kept groups only.
 *
 * sel[0..k_r) receives the chosen experts in selection order.
 */
static void orc_select(const float* key, int E, int k_r, int n_group, int topk_group, orc_kv* work,
                       int32_t* sel)
{
    int n = 0;
    if (n_group > 0) {
        int gs = E / n_group;
        int m = k_r / topk_group;
        orc_kv* groups = (orc_kv*)malloc(sizeof(orc_kv) * (size_t)n_group);
        for (int g = 0; g < n_group; ++g) {
            for (int i = 0; i < gs; ++i) {
                work[i].key = key[g * gs + i];
                work[i].idx = g * gs + i;
            }
            orc_order(work, gs);
            float acc = work[0].key;
            for (int i = 1; i < m; ++i) acc = acc + work[i].key;
            groups[g].key = acc;
            groups[g].idx = g;
        }
        orc_order(groups, n_group);
        for (int j = 0; j < topk_group; ++j) {
            int g = groups[j].idx;
            for (int i = 0; i < gs; ++i) {
                work[n].key = key[g * gs + i];
                work[n].idx = g * gs + i;
                ++n;
            }
        }
        free(groups);
    } else {
        for (int e = 0; e < E; ++e) {
            work[e].key = key[e];
            work[e].idx = e;
        }
        n = E;
    }
    orc_order(work, n);
    for (int j = 0; j < k_r; ++j) sel[j] = work[j].idx;
}

/*
 * Router forward ([TE] fused_topk_with_score_function; flowchart: score fn ->
 * top-k -> write probs + routing_map; outputs probs, routing_map and
 * intermediate_output per "Performance").
 *
 * Per token row of `logits` (T x E, fp32; bf16 logits are widened exactly by
 * the caller):
 *   s        = score_fn(x)                        (double)
 *   chosen   = top-k_r experts by key, k_r = topk - n_shared
 *   w_j      = s[chosen_j]; if renorm: w_j /= sum_j s[chosen_j] (0 if that sum is 0);
 *              then w_j *= scaling                 (READING: weights use the unbiased score)
 *   slots k_r..topk-1 hold the shared experts E..E+n_shared-1 with weight
 *   shared_weight, neither renormalised nor scaled (READING).
 * Outputs (each may be NULL):
 *   probs[T x E]        w at chosen experts, 0 elsewhere
 *   routing_map[T x E]  1 at chosen experts, 0 elsewhere
 *   intermediate[T x E] s
 *   topk_idx[T x topk], topk_w[T x topk]   in selection order, then shared slots
 */
int orc_router_fwd(int T, int E, int topk, int score_fn, int renorm, int n_group, int topk_group,
                   int n_shared, float scaling, float shared_weight, const float* logits,
                   const float* bias, double* probs, uint8_t* routing_map, double* intermediate,
                   int32_t* topk_idx, double* topk_w)
{
    int k_r = topk - n_shared;
    if (T < 0 || E < 1 || n_shared < 0 || k_r < 1 || k_r > E || !logits) return -1;
    if (score_fn != ORC_SOFTMAX && score_fn != ORC_SIGMOID) return -1;
    /* A bias or a group limit needs a selection key that the softmax reading
     * (key = logit) does not define; those combinations are rejected. */
    if (score_fn == ORC_SOFTMAX && (bias || n_group > 0)) return -1;
    if (n_group > 0) {
        if (E % n_group || topk_group < 1 || topk_group > n_group || k_r % topk_group) return -1;
        if (k_r / topk_group > E / n_group) return -1;
    }
    double* s = (double*)malloc(sizeof(double) * (size_t)E);
    float* key = (float*)malloc(sizeof(float) * (size_t)E);
    orc_kv* work = (orc_kv*)malloc(sizeof(orc_kv) * (size_t)E);
    int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * (size_t)k_r);
    for (int t = 0; t < T; ++t) {
        const float* x = logits + (size_t)t * E;
        orc_scores(score_fn, x, E, s);
        orc_keys(score_fn, x, bias, E, key);
        orc_select(key, E, k_r, n_group, topk_group, work, sel);
        double sum = 0.0;
        for (int j = 0; j < k_r; ++j) sum += s[sel[j]];
        if (probs)
            for (int e = 0; e < E; ++e) probs[(size_t)t * E + e] = 0.0;
        if (routing_map)
            for (int e = 0; e < E; ++e) routing_map[(size_t)t * E + e] = 0;
        if (intermediate)
            for (int e = 0; e < E; ++e) intermediate[(size_t)t * E + e] = s[e];
        for (int j = 0; j < k_r; ++j) {
            int e = sel[j];
            double w = s[e];
            if (renorm) w = (sum > 0.0) ? w / sum : 0.0;
            w = w * (double)scaling;
            if (probs) probs[(size_t)t * E + e] = w;
            if (routing_map) routing_map[(size_t)t * E + e] = 1;
            if (topk_idx) topk_idx[(size_t)t * topk + j] = e;
            if (topk_w) topk_w[(size_t)t * topk + j] = w;
        }
        for (int j = k_r; j < topk; ++j) {
            if (topk_idx) topk_idx[(size_t)t * topk + j] = E + (j - k_r);
            if (topk_w) topk_w[(size_t)t * topk + j] = (double)shared_weight;
        }
    }
    free(s);
    free(key);
    free(work);
    free(sel);
    return 0;
}

/*
 * Aux-loss scores forward ([TE] fused_score_for_moe_aux_loss): the score
 * function over all E experts (READING: the raw softmax or sigmoid, no bias, no
 * groups) and the routing_map of the top-k of those unbiased scores.
 */
int orc_aux_scores_fwd(int T, int E, int topk, int score_fn, const float* logits, double* scores,
                       uint8_t* routing_map)
{
    return orc_router_fwd(T, E, topk, score_fn, 0, 0, 0, 0, 1.0f, 0.0f, logits, NULL, NULL,
                          routing_map, scores, NULL, NULL);
}

/*
 * Router backward ([TE] "Two-pass fused design" of the top-k backward), the
 * chain rule through the forward above with the selection held fixed:
 *   g = dL/dprobs, s = intermediate, m = routing_map, c = scaling
 *   without renorm: ds_i = c * m_i * g_i
 *   with renorm:    A = sum_e m_e s_e,  B = sum_e m_e s_e g_e,
 *                   ds_i = (c * m_i / A) * (g_i - B / A)      (0 when A == 0)
 *   softmax:        dx_i = s_i * (ds_i - sum_j s_j ds_j)
 *   sigmoid:        dx_i = ds_i * s_i * (1 - s_i)
 * The bias and the group limit only choose experts and carry no gradient.
 */
int orc_router_bwd(int T, int E, int score_fn, int renorm, float scaling, const double* grad,
                   const double* inter, const uint8_t* routing_map, double* grad_logits)
{
    if (T < 0 || E < 1 || !grad || !inter || !routing_map || !grad_logits) return -1;
    if (score_fn != ORC_SOFTMAX && score_fn != ORC_SIGMOID) return -1;
    double* ds = (double*)malloc(sizeof(double) * (size_t)E);
    const double c = (double)scaling;
    for (int t = 0; t < T; ++t) {
        const double* g = grad + (size_t)t * E;
        const double* s = inter + (size_t)t * E;
        const uint8_t* m = routing_map + (size_t)t * E;
        double* dx = grad_logits + (size_t)t * E;
        if (renorm) {
            double A = 0.0, B = 0.0;
            for (int e = 0; e < E; ++e) {
                if (m[e]) {
                    A += s[e];
                    B += s[e] * g[e];
                }
            }
            for (int e = 0; e < E; ++e)
                ds[e] = (m[e] && A != 0.0) ? (c / A) * (g[e] - B / A) : 0.0;
        } else {
            for (int e = 0; e < E; ++e) ds[e] = m[e] ? c * g[e] : 0.0;
        }
        if (score_fn == ORC_SOFTMAX) {
            double D = 0.0;
            for (int e = 0; e < E; ++e) D += s[e] * ds[e];
            for (int e = 0; e < E; ++e) dx[e] = s[e] * (ds[e] - D);
        } else {
            for (int e = 0; e < E; ++e) dx[e] = ds[e] * s[e] * (1.0 - s[e]);
        }
    }
    free(ds);
    return 0;
}

/*
 * Aux-loss scores backward ([TE] fused_score_for_moe_aux_loss backward):
 *   softmax: dx_i = s_i * (g_i - sum_j g_j s_j)
 *   sigmoid: dx_i = g_i * s_i * (1 - s_i)
 */
int orc_aux_scores_bwd(int T, int E, int score_fn, const double* grad, const double* scores,
                       double* grad_logits)
{
    if (T < 0 || E < 1 || !grad || !scores || !grad_logits) return -1;
    if (score_fn != ORC_SOFTMAX && score_fn != ORC_SIGMOID) return -1;
    for (int t = 0; t < T; ++t) {
        const double* g = grad + (size_t)t * E;
        const double* s = scores + (size_t)t * E;
        double* dx = grad_logits + (size_t)t * E;
        if (score_fn == ORC_SOFTMAX) {
            double D = 0.0;
            for (int e = 0; e < E; ++e) D += g[e] * s[e];
            for (int e = 0; e < E; ++e) dx[e] = s[e] * (g[e] - D);
        } else {
            for (int e = 0; e < E; ++e) dx[e] = g[e] * s[e] * (1.0 - s[e]);
        }
    }
    return 0;
}

/*
 * Sorting ([FLY] moe_sorting; layout pinned by [GEMM]).
 *
 * Input: topk_idx[T x topk] (expert of each (token, slot) pair) and
 * topk_w[T x topk]; E_tot experts; block size block_m.
 *   cnt[e]  = number of pairs routed to expert e (ids outside [0, E_tot) are
 *             dropped and counted in the return value)
 *   pad[e]  = ceil(cnt[e] / block_m) * block_m        (0 for an empty expert)
 *   off[e]  = sum_{e' < e} pad[e']
 *   num_tokens_post_pad = sum_e pad[e]
 *   sorted_token_ids[off[e] + r] = t*topk + j for the r-th pair of expert e in
 *       ascending (t, j) order (READING: stable in the flat index);
 *       positions off[e]+cnt[e] .. off[e]+pad[e]-1 hold the sentinel T*topk
 *       (one past the last valid row, so it can never alias a real row)
 *   sorted_weights: the pair's weight, 0 at sentinel positions
 *   expert_ids[b] = e for every block b of expert e's range.
 * Experts appear in ascending id order. Only [0, num_tokens_post_pad) and
 * [0, num_tokens_post_pad / block_m) are written.
 *
 * Returns the number of dropped pairs (>= 0), or -1 on bad arguments.
 */
size_t orc_sort_capacity(int T, int topk, int E_tot, int block_m)
{
    size_t n = (size_t)T * (size_t)topk;
    size_t nonempty = (size_t)E_tot < n ? (size_t)E_tot : n;
    return n + nonempty * (size_t)(block_m - 1);
}

int orc_sort(const int32_t* topk_idx, const float* topk_w, int T, int topk, int E_tot, int block_m,
             int32_t* sorted_token_ids, float* sorted_weights, int32_t* expert_ids,
             int32_t* num_tokens_post_pad)
{
    if (T < 0 || topk < 1 || E_tot < 1 || block_m < 1 || !topk_idx || !sorted_token_ids ||
        !expert_ids || !num_tokens_post_pad)
        return -1;
    const int64_t n = (int64_t)T * topk;
    int64_t* cnt = (int64_t*)calloc((size_t)E_tot, sizeof(int64_t));
    int dropped = 0;
    for (int64_t f = 0; f < n; ++f) {
        int32_t e = topk_idx[f];
        if (e < 0 || e >= E_tot)
            ++dropped;
        else
            ++cnt[e];
    }
    int64_t pos = 0;
    for (int e = 0; e < E_tot; ++e) {
        int64_t pad = (cnt[e] + block_m - 1) / block_m * block_m;
        int64_t start = pos;
        for (int64_t f = 0; f < n; ++f) {
            if (topk_idx[f] == e) {
                sorted_token_ids[pos] = (int32_t)f;
                if (sorted_weights) sorted_weights[pos] = topk_w ? topk_w[f] : 0.0f;
                ++pos;
            }
        }
        for (; pos < start + pad; ++pos) {
            sorted_token_ids[pos] = (int32_t)n;
            if (sorted_weights) sorted_weights[pos] = 0.0f;
        }
        for (int64_t b = start / block_m; b < (start + pad) / block_m; ++b) expert_ids[b] = e;
    }
    *num_tokens_post_pad = (int32_t)pos;
    free(cnt);
    return dropped;
}

/* ------------------------------------------------------------------------- */
/* Aux-loss scalar ([TE] fused_moe_aux_loss).                                */
/* ------------------------------------------------------------------------- */
/*
 * READING. [TE] names the fused_moe_aux_loss kernel (it consumes the scores and
 * routing map of fused_score_for_moe_aux_loss) but prints no formula. It is
 * read as the load-balancing loss of switch-style routing (Fedus, Zoph and
 * Shazeer, "Switch Transformers", 2021, the auxiliary loss of section 2.2):
 * with f_e the fraction of the routed slots that went to expert e and P_e the
 * mean router probability of expert e,
 *     loss = coeff * E * sum_e f_e * P_e,
 *     f_e  = tokens_per_expert[e] / (topk * N),
 *     P_e  = (sum_t probs[t][e]) / N,
 * where N = total_num_tokens, the number of tokens the counts and the
 * probabilities were taken over (it may exceed the T rows given here when the
 * tokens are spread over several devices). tokens_per_expert is a count, so
 * the gradient flows only through probs:
 *     d loss / d probs[t][e] = coeff * E * f_e / N * grad_loss.
 */

/* tokens_per_expert[e] = number of rows t with routing_map[t][e] != 0. */
int orc_tokens_per_expert(int T, int E, const uint8_t* routing_map, int32_t* tokens_per_expert)
{
    if (T < 0 || E < 1 || (T > 0 && !routing_map) || !tokens_per_expert) return -1;
    for (int e = 0; e < E; ++e) {
        int64_t c = 0;
        for (int t = 0; t < T; ++t) c += routing_map[(size_t)t * E + e] != 0;
        tokens_per_expert[e] = (int32_t)c;
    }
    return 0;
}

int orc_aux_loss_fwd(int T, int E, int topk, double coeff, int64_t total_num_tokens, const double* probs,
                     const int32_t* tokens_per_expert, double* loss)
{
    if (T < 0 || E < 1 || topk < 1 || total_num_tokens < 1 || (T > 0 && !probs) || !tokens_per_expert ||
        !loss)
        return -1;
    const double N = (double)total_num_tokens;
    double acc = 0.0;
    for (int e = 0; e < E; ++e) {
        double colsum = 0.0;
        for (int t = 0; t < T; ++t) colsum += probs[(size_t)t * E + e];
        const double f = (double)tokens_per_expert[e] / ((double)topk * N);
        const double P = colsum / N;
        acc += f * P;
    }
    *loss = coeff * (double)E * acc;
    return 0;
}

int orc_aux_loss_bwd(int T, int E, int topk, double coeff, int64_t total_num_tokens,
                     const int32_t* tokens_per_expert, double grad_loss, double* grad_probs)
{
    if (T < 0 || E < 1 || topk < 1 || total_num_tokens < 1 || !tokens_per_expert || (T > 0 && !grad_probs))
        return -1;
    const double N = (double)total_num_tokens;
    for (int e = 0; e < E; ++e) {
        const double f = (double)tokens_per_expert[e] / ((double)topk * N);
        const double g = coeff * (double)E * f / N * grad_loss;
        for (int t = 0; t < T; ++t) grad_probs[(size_t)t * E + e] = g;
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Near ties at the selection boundary (informational; not a step of the     */
/* method). Per token, the selection keys in double (softmax: the logit;     */
/* sigmoid: 1/(1 + e^-x) plus the bias) sorted descending, and              */
/*   gap[t] = (key_(k_r) - key_(k_r+1)) / ulp_fp32(key_(k_r+1)),             */
/* the distance between the last key taken and the first left out, in fp32   */
/* ulps at the latter's magnitude. A token with a gap of a few ulps is one   */
/* whose selected set another fp32 rounding of its keys could change: the    */
/* rows where bit-exact agreement of the selections says the most.           */
/* k_r >= E: gap = -1 (no key is left out).                                  */
/* ------------------------------------------------------------------------- */
static int orc_desc_double(const void* a, const void* b)
{
    const double x = *(const double*)a, y = *(const double*)b;
    return (x < y) - (x > y);
}

/* spacing of fp32 values around |v| (the subnormal spacing below FLT_MIN) */
static double orc_ulp_f32(double v)
{
    v = fabs(v);
    if (v < ldexp(1.0, -126)) return ldexp(1.0, -149);
    int ex;
    frexp(v, &ex); /* v = f * 2^ex, 0.5 <= f < 1: fp32 spacing 2^(ex - 24) */
    return ldexp(1.0, ex - 24);
}

int orc_near_tie_gaps(int T, int E, int k_r, int score_fn, const float* logits, const float* bias, double* gap)
{
    if (T < 0 || E < 1 || k_r < 1 || (T > 0 && (!logits || !gap))) return -1;
    double* key = (double*)malloc(sizeof(double) * (size_t)E);
    if (!key) return -1;
    for (int t = 0; t < T; ++t) {
        const float* x = logits + (size_t)t * E;
        if (k_r >= E) {
            gap[t] = -1.0;
            continue;
        }
        for (int e = 0; e < E; ++e)
            key[e] = score_fn == ORC_SOFTMAX ? (double)x[e]
                                              : 1.0 / (1.0 + exp(-(double)x[e])) + (bias ? (double)bias[e] : 0.0);
        qsort(key, (size_t)E, sizeof(double), orc_desc_double);
        gap[t] = (key[k_r - 1] - key[k_r]) / orc_ulp_f32(key[k_r]);
    }
    free(key);
    return 0;
}
