/*
 * moe_oracle.c -- plain CPU oracle of the MoE feed-forward layer.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load or call this code.  It shares no code,
 * header, table or helper with the CUDA library and never calls it.
 *
 * Source: "NPU HunyuanImage-3.0模型推理优化实践" (cf-1.com/news/2296994),
 * which describes one MoE layer of HunyuanImage-3.0:
 *   - "RmsNorm算子优化": RMSNorm, i.e. LayerNorm without the mean subtraction;
 *   - "消除gate计算冗余cast算子": the gate is an fp32 linear layer on the
 *     hidden states cast to float (autocast switched off);
 *   - "MoE EP优化": GatingTopK, then InitRouting (which expert each token
 *     goes to), expert compute, FinalizeRouting;
 *   - "MoE TP优化 / 计算分解": each expert computes
 *     x = down(SiLU(gate(x)) * up(x)); gate and up are merged into one weight
 *     w13 and the SwiGLU step chunks the last dim in two halves and returns
 *     SiLU(x[0]) * x[1];
 *   - "GMM使能&&Routing优化": init_routing sorts the tokens by expert,
 *     compute_expert_tokens counts the tokens of every expert, one grouped
 *     matmul serves all experts, finalize_routing puts the expert outputs back
 *     in token order and forms the weighted sum;
 *   - "MoE多流并行优化": a shared expert is computed beside the routed ones
 *     and summed in.
 *
 * Readings where the page is silent (each is listed in the design notes):
 *   - RMSNorm: r = 1/sqrt(mean(x^2) + eps) in fp32, where the sum of squares
 *     is the exact sum of the bf16 squares rounded once to fp32 (nearest,
 *     ties to even), so it does not depend on a summation order;
 *     xn = bf16((x * r) * gamma).
 *   - Gate: every logit is an fp32 dot product accumulated in ascending h with
 *     one fused multiply-add per term, plus an optional per-expert offset.
 *     Routing decisions are taken on these fp32 logits (the page's precision).
 *   - Top-k by logit, descending, equal logits to the lower expert index;
 *     weights = softmax probabilities of the chosen experts, renormalised to
 *     sum 1 (in double here).
 *   - Routing is the stable counting sort of the T*k assignments a = t*k + j
 *     by expert.
 *   - Expert MLP: fp64 sums of the exact bf16 products; act and the routed
 *     expert output are rounded to bf16 (the grouped matmul's output type);
 *     the shared expert output enters the final sum unrounded.  A second
 *     reading keeps the routed expert output unrounded too (the library's
 *     fp32-y mode, where the down matmul's accumulator goes straight into the
 *     weighted sum); only the SwiGLU output is then rounded to bf16.
 *   - Finalize: out[t] = sum_j w[t,j] * y[row(t,j)] + shared[t], in double.
 *
 * bf16 tensors are passed as uint16 bit patterns.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef uint16_t bf16_t;

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_BAD_EXPERT = 2, ORACLE_NOMEM = 3 };

static float bf16_to_float(bf16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a double to the nearest bf16, ties to even, in one step (no detour
 * through float, which would round twice). */
static bf16_t bf16_from_double(double d)
{
    if (isnan(d))
        return 0x7FC0;
    const uint16_t sign = signbit(d) ? 0x8000 : 0;
    const double a = fabs(d);
    if (a == 0.0)
        return sign;
    double q;
    if (a < 0x1p-126) {
        /* bf16 subnormals are multiples of 2^-133 */
        q = nearbyint(a * 0x1p133) * 0x1p-133;
    } else {
        int e;
        const double m = frexp(a, &e);          /* a = m * 2^e, m in [0.5, 1) */
        q = ldexp(nearbyint(ldexp(m, 8)), e - 8); /* keep 8 significant bits */
    }
    if (q > 0x1.FEp127)                          /* beyond the largest bf16 */
        return sign | 0x7F80;
    const float f = (float)q;                    /* exact */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------ */
/* Sum of squares of a bf16 row, exact, rounded once to fp32 (nearest, ties  */
/* to even).  A finite bf16 value is m * 2^(E - 134) with m its 8-bit       */
/* significand (implicit bit included) and E = max(biased exponent, 1), so  */
/* its square is m^2 * 2^(2E - 268): an integer m^2 < 2^16 shifted left by   */
/* 2E - 2 bits in a fixed-point number whose unit is 2^-266.  The squares    */
/* are added into such a number held in 64-bit limbs (2E - 2 <= 506, plus    */
/* 16 bits of m^2 and 31 bits of carries fit 12 limbs), which is then        */
/* rounded to 24 significant bits, or to a multiple of 2^-149 (bit 117) in   */
/* fp32's subnormal range.  A row holding an infinity or a NaN gives the     */
/* plain fp32 sum (inf or NaN).                                             */
#define SS_LIMBS 12
static float sumsq_exact_rn(const bf16_t *x, int64_t H)
{
    uint64_t acc[SS_LIMBS];
    memset(acc, 0, sizeof acc);
    for (int64_t h = 0; h < H; ++h) {
        const int e = (x[h] >> 7) & 0xFF;
        if (e == 0xFF) {
            float s = 0.0f;
            for (int64_t i = 0; i < H; ++i)
                s += bf16_to_float(x[i]) * bf16_to_float(x[i]);
            return s;
        }
        const uint64_t m = (uint64_t)(x[h] & 0x7F) | (e ? 0x80u : 0u);
        const int sh = 2 * (e ? e : 1) - 2;
        const int li = sh / 64, bo = sh % 64;
        const uint64_t sq = m * m;
        /* sq << bo spans limbs li and li + 1 */
        uint64_t add[2];
        add[0] = sq << bo;
        add[1] = bo ? sq >> (64 - bo) : 0;
        uint64_t carry = 0;
        for (int j = li; j < SS_LIMBS; ++j) {
            const uint64_t a = (j - li < 2) ? add[j - li] : 0;
            const uint64_t old = acc[j];
            acc[j] = old + a + carry;
            carry = (acc[j] < old || (carry && acc[j] == old)) ? 1 : 0;
            if (j - li >= 1 && !carry)
                break;
        }
    }
    /* the highest set bit */
    int top = -1;
    for (int j = SS_LIMBS - 1; j >= 0 && top < 0; --j)
        for (int b = 63; b >= 0; --b)
            if ((acc[j] >> b) & 1) {
                top = j * 64 + b;
                break;
            }
    if (top < 0)
        return 0.0f;
    int lsb = top - 23;            /* keep 24 significant bits */
    if (lsb < 117)
        lsb = 117;                 /* fp32 subnormals: multiples of 2^-149 */
#define SS_BIT(i) ((int)((acc[(i) / 64] >> ((i) % 64)) & 1))
    uint64_t q = 0;
    for (int i = top; i >= lsb; --i)
        q = (q << 1) | (uint64_t)SS_BIT(i);
    /* the part below lsb against half of one unit of lsb */
    int round_up = 0;
    if (lsb > 0 && SS_BIT(lsb - 1)) {
        int rest = 0;
        for (int i = lsb - 2; i >= 0 && !rest; --i)
            rest = SS_BIT(i);
        round_up = rest || (q & 1);
    }
#undef SS_BIT
    q += (uint64_t)round_up;
    /* q * 2^(lsb - 266): exact in double; the cast to float is exact too,
       unless it overflows to infinity */
    return (float)ldexp((double)q, lsb - 266);
}

/* The row sums of squares as the RMSNorm takes them (test access). */
int oracle_sumsq(const bf16_t *x, int64_t T, int64_t H, float *ss)
{
    if (!x || !ss || T < 0 || H <= 0)
        return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        ss[t] = sumsq_exact_rn(x + t * H, H);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* RMSNorm ("RmsNorm算子优化"): xn = x / sqrt(mean(x^2) + eps) * gamma.       */
/* gamma may be NULL (all ones).                                            */
int oracle_rmsnorm(const bf16_t *x, const bf16_t *gamma, int64_t T, int64_t H,
                   float eps, bf16_t *xn)
{
    if (!x || !xn || T < 0 || H <= 0)
        return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const bf16_t *xr = x + t * H;
        const float ss = sumsq_exact_rn(xr, H);
        const float mean = ss / (float)H;
        const float r = 1.0f / sqrtf(mean + eps);
        for (int64_t h = 0; h < H; ++h) {
            float v = bf16_to_float(xr[h]) * r;
            if (gamma)
                v = v * bf16_to_float(gamma[h]);
            xn[t * H + h] = bf16_from_double((double)v);
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* fp32 gate ("消除gate计算冗余cast算子"): logits = float(hidden) @ wg^T       */
/* (+ bias).  wg is [E, H] fp32, bias [E] fp32 or NULL.                      */
int oracle_gate_logits(const bf16_t *xs, const float *wg, const float *bias,
                       int64_t T, int64_t H, int64_t E, float *logits)
{
    if (!xs || !wg || !logits || T < 0 || H <= 0 || E <= 0)
        return ORACLE_BAD_ARG;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t e = 0; e < E; ++e) {
            float acc = 0.0f;
            for (int64_t h = 0; h < H; ++h)
                acc = fmaf(bf16_to_float(xs[t * H + h]), wg[e * H + h], acc);
            if (bias)
                acc = acc + bias[e];
            logits[t * E + e] = acc;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* GatingTopK ("MoE EP优化"): softmax over the E logits of a token, the k     */
/* largest, and (renorm != 0) their probabilities divided by their sum.     */
/* Slot j = 0 holds the largest logit; equal logits go to the lower index.  */
int oracle_topk_softmax(const float *logits, int64_t T, int64_t E, int64_t k,
                        int renorm, int32_t *topk_idx, float *topk_w)
{
    if (!logits || !topk_idx || !topk_w || T < 0 || E <= 0 || k < 1 || k > E)
        return ORACLE_BAD_ARG;
    int status = ORACLE_OK;
#pragma omp parallel
    {
        unsigned char *taken = (unsigned char *)malloc((size_t)E);
        if (!taken) {
#pragma omp atomic write
            status = ORACLE_NOMEM;
        }
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            if (!taken)
                continue;
            const float *l = logits + t * E;
            memset(taken, 0, (size_t)E);
            for (int64_t j = 0; j < k; ++j) {
                int64_t best = -1;
                for (int64_t e = 0; e < E; ++e)
                    if (!taken[e] && (best < 0 || l[e] > l[best]))
                        best = e;
                taken[best] = 1;
                topk_idx[t * k + j] = (int32_t)best;
            }
            /* softmax with the row maximum (= logit of slot 0) subtracted */
            const double m = (double)l[topk_idx[t * k]];
            double den = 0.0;
            if (renorm) {
                for (int64_t j = 0; j < k; ++j)
                    den += exp((double)l[topk_idx[t * k + j]] - m);
            } else {
                for (int64_t e = 0; e < E; ++e)
                    den += exp((double)l[e] - m);
            }
            for (int64_t j = 0; j < k; ++j)
                topk_w[t * k + j] =
                    (float)(exp((double)l[topk_idx[t * k + j]] - m) / den);
        }
        free(taken);
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* init_routing ("GMM使能&&Routing优化": sort the tokens by expert).          */
/* Assignment a = t*k + j goes to expert topk_idx[a].  Counting sort, stable */
/* in a:                                                                    */
/*   counts[e]  = number of assignments to e, offsets = exclusive scan      */
/*   row_idx[a] = offsets[e] + #{a' < a : topk_idx[a'] == e}                */
/*   src_token[row_idx[a]] = a / k,  sorted_ids[row_idx[a]] = e             */
/* sorted_ids may be NULL.                                                  */
int oracle_init_routing(const int32_t *topk_idx, int64_t T, int64_t k, int64_t E,
                        int32_t *row_idx, int32_t *src_token, int32_t *sorted_ids,
                        int32_t *counts, int32_t *offsets)
{
    if (!topk_idx || !row_idx || !src_token || !counts || !offsets || T < 0 ||
        k < 1 || E <= 0)
        return ORACLE_BAD_ARG;
    const int64_t N = T * k;
    for (int64_t a = 0; a < N; ++a)
        if (topk_idx[a] < 0 || topk_idx[a] >= E)
            return ORACLE_BAD_EXPERT;
    for (int64_t e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t a = 0; a < N; ++a)
        counts[topk_idx[a]] += 1;
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    if (!fill)
        return ORACLE_NOMEM;
    for (int64_t a = 0; a < N; ++a) {
        const int32_t e = topk_idx[a];
        const int32_t row = offsets[e] + fill[e]++;
        row_idx[a] = row;
        src_token[row] = (int32_t)(a / k);
        if (sorted_ids)
            sorted_ids[row] = e;
    }
    free(fill);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* compute_expert_tokens ("GMM使能&&Routing优化": tokens per expert), from    */
/* the expert ids of the sorted rows.                                       */
int oracle_expert_tokens(const int32_t *ids, int64_t n, int64_t E, int32_t *counts,
                         int32_t *offsets)
{
    if ((!ids && n > 0) || !counts || !offsets || n < 0 || E <= 0)
        return ORACLE_BAD_ARG;
    for (int64_t e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= E)
            return ORACLE_BAD_EXPERT;
        counts[ids[i]] += 1;
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* The data half of init_routing: expanded_x[r] = xs[src_token[r]].          */
int oracle_permute(const bf16_t *xs, const int32_t *src_token, int64_t n, int64_t H,
                   bf16_t *expanded_x)
{
    if (!xs || !src_token || !expanded_x || n < 0 || H <= 0)
        return ORACLE_BAD_ARG;
    for (int64_t r = 0; r < n; ++r)
        memcpy(expanded_x + r * H, xs + (int64_t)src_token[r] * H,
               (size_t)H * sizeof(bf16_t));
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* One expert's FFN ("MoE TP优化 / 计算分解"): x = down(SiLU(gate(x)) * up(x)) */
/* on n rows.  w13 is [2I, H] (rows 0..I-1 gate, I..2I-1 up), w2 is [H, I].  */
/*   g = xe . w13[i],  u = xe . w13[I+i]        (fp64 sums of exact products) */
/*   act[i] = bf16(SiLU(g) * u),  SiLU(g) = g / (1 + exp(-g))                */
/*   y[c]   = sum_i act[i] * w2[c, i]                                        */
/* y is returned rounded to bf16 (y_bf16) and/or unrounded (y_f64); either   */
/* may be NULL, act may be NULL.                                            */
int oracle_expert_mlp(const bf16_t *xe, int64_t n, const bf16_t *w13,
                      const bf16_t *w2, int64_t H, int64_t I, bf16_t *act,
                      bf16_t *y_bf16, double *y_f64)
{
    if ((!xe && n > 0) || !w13 || !w2 || n < 0 || H <= 0 || I <= 0)
        return ORACLE_BAD_ARG;
    bf16_t *a = act;
    bf16_t *own = NULL;
    if (!a) {
        own = (bf16_t *)malloc((size_t)(n > 0 ? n : 1) * (size_t)I * sizeof(bf16_t));
        if (!own)
            return ORACLE_NOMEM;
        a = own;
    }
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t i = 0; i < I; ++i) {
            const bf16_t *xr = xe + r * H;
            const bf16_t *wgate = w13 + i * H;
            const bf16_t *wup = w13 + (I + i) * H;
            double g = 0.0, u = 0.0;
            for (int64_t h = 0; h < H; ++h) {
                const double xv = (double)bf16_to_float(xr[h]);
                g += xv * (double)bf16_to_float(wgate[h]);
                u += xv * (double)bf16_to_float(wup[h]);
            }
            const double silu = g / (1.0 + exp(-g));
            a[r * I + i] = bf16_from_double(silu * u);
        }
    }
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t c = 0; c < H; ++c) {
            const bf16_t *ar = a + r * I;
            const bf16_t *wr = w2 + c * I;
            double y = 0.0;
            for (int64_t i = 0; i < I; ++i)
                y += (double)bf16_to_float(ar[i]) * (double)bf16_to_float(wr[i]);
            if (y_bf16)
                y_bf16[r * H + c] = bf16_from_double(y);
            if (y_f64)
                y_f64[r * H + c] = y;
        }
    }
    free(own);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Grouped matmul ("GMM使能&&Routing优化"): group g owns the sorted rows      */
/* [offsets[g], offsets[g+1]) of expanded_x and uses w13[g], w2[g].          */
int oracle_grouped_mlp(const bf16_t *expanded_x, const int32_t *offsets, int64_t G,
                       const bf16_t *w13, const bf16_t *w2, int64_t H, int64_t I,
                       bf16_t *act, bf16_t *y)
{
    if (!expanded_x || !offsets || !w13 || !w2 || !act || !y || G <= 0)
        return ORACLE_BAD_ARG;
    for (int64_t g = 0; g < G; ++g) {
        const int64_t r0 = offsets[g], r1 = offsets[g + 1];
        if (r1 < r0)
            return ORACLE_BAD_ARG;
        if (r1 == r0)
            continue;
        const int rc = oracle_expert_mlp(expanded_x + r0 * H, r1 - r0,
                                         w13 + g * 2 * I * H, w2 + g * H * I, H, I,
                                         act + r0 * I, y + r0 * H, NULL);
        if (rc != ORACLE_OK)
            return rc;
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* finalize_routing ("GMM使能&&Routing优化": put expert outputs back in token */
/* order and form the weighted sum) plus the shared expert ("MoE多流并行优化"):*/
/*   out[t, c] = sum_{j<k} w[t, j] * y[row_idx[t*k+j], c] + shared[t, c]     */
/* shared may be NULL.                                                      */
int oracle_finalize(const bf16_t *y_exp, const int32_t *row_idx, const float *topk_w,
                    const double *shared, int64_t T, int64_t H, int64_t k, double *out)
{
    if (!y_exp || !row_idx || !topk_w || !out || T < 0 || H <= 0 || k < 1)
        return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t c = 0; c < H; ++c) {
            double s = 0.0;
            for (int64_t j = 0; j < k; ++j)
                s += (double)topk_w[t * k + j] *
                     (double)bf16_to_float(y_exp[(int64_t)row_idx[t * k + j] * H + c]);
            if (shared)
                s += shared[t * H + c];
            out[t * H + c] = s;
        }
    }
    return ORACLE_OK;
}

/* The same weighted sum over unrounded routed rows y_exp [T*k, H] double    */
/* (the fp32-y reading: no bf16 rounding of the expert outputs).            */
int oracle_finalize_f64(const double *y_exp, const int32_t *row_idx, const float *topk_w,
                        const double *shared, int64_t T, int64_t H, int64_t k, double *out)
{
    if (!y_exp || !row_idx || !topk_w || !out || T < 0 || H <= 0 || k < 1)
        return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t c = 0; c < H; ++c) {
            double s = 0.0;
            for (int64_t j = 0; j < k; ++j)
                s += (double)topk_w[t * k + j] * y_exp[(int64_t)row_idx[t * k + j] * H + c];
            if (shared)
                s += shared[t * H + c];
            out[t * H + c] = s;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* The whole layer for a list of tokens.  A token's output depends only on  */
/* its own row and the weights, so any subset is exact for those tokens.    */
/*   x [T,H] bf16; gamma [H] bf16 or NULL (no RMSNorm when rmsnorm == 0);    */
/*   wg [E,H] fp32; bias [E] or NULL; w13 [E,2I,H]; w2 [E,H,I];             */
/*   w13_s [2I_s,H], w2_s [H,I_s] or NULL (no shared expert);               */
/*   tokens [n_tok] (NULL = 0..T-1, n_tok = T).                             */
/* Outputs: out [n_tok,H] double; idx/w [n_tok,k] (may be NULL);            */
/*   y_out [n_tok,k,H] bf16 (may be NULL): each slot's routed expert output,  */
/*   rounded to bf16.                                                       */
/*   out_yf [n_tok,H] double (may be NULL): the same layer in the fp32-y    */
/*   reading, the routed expert outputs entering the weighted sum unrounded. */
int oracle_layer_tokens(const bf16_t *x, int64_t T, int64_t H, int64_t E, int64_t k,
                        int64_t I, int64_t I_s, int rmsnorm, float eps, int renorm,
                        const bf16_t *gamma, const float *wg, const float *bias,
                        const bf16_t *w13, const bf16_t *w2, const bf16_t *w13_s,
                        const bf16_t *w2_s, const int32_t *tokens, int64_t n_tok,
                        double *out, int32_t *idx_out, float *w_out, bf16_t *y_out,
                        double *out_yf)
{
    if (!x || !wg || !w13 || !w2 || !out || H <= 0 || E <= 0 || k < 1 || k > E ||
        I <= 0 || I_s < 0 || (I_s > 0 && (!w13_s || !w2_s)))
        return ORACLE_BAD_ARG;
    if (!tokens)
        n_tok = T;
    int rc = ORACLE_OK;
    bf16_t *xrow = (bf16_t *)malloc((size_t)H * sizeof(bf16_t));
    float *logits = (float *)malloc((size_t)E * sizeof(float));
    int32_t *idx = (int32_t *)malloc((size_t)k * sizeof(int32_t));
    float *w = (float *)malloc((size_t)k * sizeof(float));
    bf16_t *yb = (bf16_t *)malloc((size_t)H * sizeof(bf16_t));
    double *ys = (double *)malloc((size_t)H * sizeof(double));
    double *yr = (double *)malloc((size_t)H * sizeof(double));
    if (!xrow || !logits || !idx || !w || !yb || !ys || !yr) {
        rc = ORACLE_NOMEM;
        goto done;
    }
    for (int64_t n = 0; n < n_tok; ++n) {
        const int64_t t = tokens ? tokens[n] : n;
        if (t < 0 || t >= T) {
            rc = ORACLE_BAD_ARG;
            goto done;
        }
        if (rmsnorm)
            rc = oracle_rmsnorm(x + t * H, gamma, 1, H, eps, xrow);
        else
            memcpy(xrow, x + t * H, (size_t)H * sizeof(bf16_t));
        if (rc)
            goto done;
        if ((rc = oracle_gate_logits(xrow, wg, bias, 1, H, E, logits)))
            goto done;
        if ((rc = oracle_topk_softmax(logits, 1, E, k, renorm, idx, w)))
            goto done;
        double *o = out + n * H;
        double *of = out_yf ? out_yf + n * H : NULL;
        for (int64_t c = 0; c < H; ++c)
            o[c] = 0.0;
        if (of)
            for (int64_t c = 0; c < H; ++c)
                of[c] = 0.0;
        for (int64_t j = 0; j < k; ++j) {
            const int64_t e = idx[j];
            if ((rc = oracle_expert_mlp(xrow, 1, w13 + e * 2 * I * H, w2 + e * H * I,
                                        H, I, NULL, yb, yr)))
                goto done;
            if (y_out)
                memcpy(y_out + (n * k + j) * H, yb, (size_t)H * sizeof(bf16_t));
            for (int64_t c = 0; c < H; ++c)
                o[c] += (double)w[j] * (double)bf16_to_float(yb[c]);
            if (of)
                for (int64_t c = 0; c < H; ++c)
                    of[c] += (double)w[j] * yr[c];
        }
        if (I_s > 0) {
            if ((rc = oracle_expert_mlp(xrow, 1, w13_s, w2_s, H, I_s, NULL, NULL, ys)))
                goto done;
            for (int64_t c = 0; c < H; ++c)
                o[c] += ys[c];
            if (of)
                for (int64_t c = 0; c < H; ++c)
                    of[c] += ys[c];
        }
        if (idx_out)
            memcpy(idx_out + n * k, idx, (size_t)k * sizeof(int32_t));
        if (w_out)
            memcpy(w_out + n * k, w, (size_t)k * sizeof(float));
    }
done:
    free(xrow);
    free(logits);
    free(idx);
    free(w);
    free(yb);
    free(ys);
    free(yr);
    return rc;
}

/* Helpers the tests use to move bf16 data in and out of the oracle. */
void oracle_bf16_round(const double *in, int64_t n, bf16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = bf16_from_double(in[i]);
}

void oracle_bf16_to_float(const bf16_t *in, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = bf16_to_float(in[i]);
}

/* ------------------------------------------------------------------------ */
/* EP DoubleRouting, local steps ("MoE EP优化"): after the token all_to_all a */
/* rank holds R received rows, grouped by source rank r = 0..ep-1, and within */
/* a source rank ordered by local expert (each rank sent its rows sorted by */
/* expert).  counts[r*E_local + e] = rows from rank r for local expert e.     */
/*                                                                          */
/* LocalRerouting ("MoE EP优化"): reorder a rank's received rows            */
/* by local expert, source rank second, arrival order third:                 */
/*   local_x[d] = recv_x[local_src[d]],                                      */
/*   local_counts[e] = sum_r counts[r][e], local_offsets = exclusive scan.   */
/* Rows past sum(counts) are left alone.                                     */
int oracle_local_rerouting(const bf16_t *recv_x, const int32_t *counts, int64_t ep,
                           int64_t E_local, int64_t R, int64_t H, bf16_t *local_x,
                           int32_t *local_src, int32_t *local_counts, int32_t *local_offsets)
{
    if (!counts || !local_src || !local_counts || !local_offsets || ep <= 0 || E_local <= 0 ||
        R < 0 || H < 0)
        return ORACLE_BAD_ARG;
    int64_t total = 0;
    for (int64_t i = 0; i < ep * E_local; ++i) {
        if (counts[i] < 0)
            return ORACLE_BAD_ARG;
        total += counts[i];
    }
    if (total > R)
        return ORACLE_BAD_ARG;
    for (int64_t e = 0; e < E_local; ++e) {
        local_counts[e] = 0;
        for (int64_t r = 0; r < ep; ++r)
            local_counts[e] += counts[r * E_local + e];
    }
    local_offsets[0] = 0;
    for (int64_t e = 0; e < E_local; ++e)
        local_offsets[e + 1] = local_offsets[e] + local_counts[e];
    /* walk the received rows in arrival order, placing each block */
    int64_t src = 0;
    for (int64_t r = 0; r < ep; ++r) {
        for (int64_t e = 0; e < E_local; ++e) {
            int64_t dst = local_offsets[e];
            for (int64_t rr = 0; rr < r; ++rr)
                dst += counts[rr * E_local + e];
            if (dst + counts[r * E_local + e] > local_offsets[e + 1])
                return ORACLE_BAD_ARG;       /* would leave expert e's rows */
            for (int64_t i = 0; i < counts[r * E_local + e]; ++i) {
                local_src[dst + i] = (int32_t)(src + i);
                if (local_x && recv_x)
                    memcpy(local_x + (dst + i) * H, recv_x + (src + i) * H,
                           (size_t)H * sizeof(bf16_t));
            }
            src += counts[r * E_local + e];
        }
    }
    return ORACLE_OK;
}

/* LocalFinalizeRerouting ("MoE EP优化"): put the expert                    */
/* outputs back in the received order: recv_y[local_src[d]] = local_y[d].    */
int oracle_local_finalize_rerouting(const bf16_t *local_y, const int32_t *local_src, int64_t n,
                                    int64_t H, bf16_t *recv_y)
{
    if ((!local_y || !local_src || !recv_y) && n > 0)
        return ORACLE_BAD_ARG;
    for (int64_t d = 0; d < n; ++d)
        memcpy(recv_y + (int64_t)local_src[d] * H, local_y + d * H, (size_t)H * sizeof(bf16_t));
    return ORACLE_OK;
}
