/*
 * colibri_oracle.c -- plain, slow CPU oracle for one routed MoE FFN layer.
 *
 * TEST INFRASTRUCTURE: see colibri_oracle.h for who may use it, the data
 * layouts and the pages each step follows. Built with
 *   gcc -std=c99 -O2 -ffp-contract=off -fno-fast-math -shared -fPIC
 * so that every fp32 operation below rounds once, as written.
 */
#include "colibri_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---- int4 unpacking ---------------------------------------------------------
 * Offset-binary nibbles, low nibble first. The pages give the container only as
 * "int4 group-scaled" (aifrontierpost tutorial, "Step 3 -- Get a model"); the
 * nibble order and the +8 offset are this layer's reading, chosen because the
 * pages' CPU kernel multiplies unsigned bytes by signed bytes (AVX2 maddubs,
 * integer dot-product row of the dashen-tech "Points techniques cles" table). */
void orc_unpack_int4(const uint8_t *packed, int64_t nbytes, int8_t *q)
{
    for (int64_t j = 0; j < nbytes; ++j) {
        q[2 * j] = (int8_t)((int)(packed[j] & 0x0F) - 8);
        q[2 * j + 1] = (int8_t)((int)(packed[j] >> 4) - 8);
    }
}

/* ---- q8 activation quantiser ------------------------------------------------
 * Symmetric absmax int8 per `group` (32, or 64 for the pages' gs64 container)
 * consecutive elements of a row, in fp32: d = amax / 127, q = clamp(roundf(x / d),
 * -127, 127), roundf rounding halves away from zero; an all-zero group gets d = 0
 * and zero codes. */
static int group_ok(int group)
{
    return group == 32 || group == 64;
}

int orc_q8_quantize_g(const float *x, int64_t rows, int64_t cols, int group, int8_t *q, float *scale)
{
    if (!group_ok(group) || rows < 0 || cols < 0 || cols % group != 0)
        return -1;
    const int64_t ng = cols / group;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < ng; ++g) {
            const float *xg = x + r * cols + g * group;
            int8_t *qg = q + r * cols + g * group;
            float amax = 0.0f;
            for (int k = 0; k < group; ++k) {
                float a = fabsf(xg[k]);
                if (a > amax)
                    amax = a;
            }
            float d = amax / 127.0f;
            scale[r * ng + g] = d;
            for (int k = 0; k < group; ++k) {
                if (d == 0.0f) {
                    qg[k] = 0;
                    continue;
                }
                float v = roundf(xg[k] / d);
                if (v > 127.0f)
                    v = 127.0f;
                if (v < -127.0f)
                    v = -127.0f;
                qg[k] = (int8_t)v;
            }
        }
    }
    return 0;
}

int orc_q8_quantize(const float *x, int64_t rows, int64_t cols, int8_t *q, float *scale)
{
    return orc_q8_quantize_g(x, rows, cols, ORC_GROUP, q, scale);
}

/* ---- router logits ----------------------------------------------------------
 * l = x . Wr[e] on the unquantised fp32 activations. The pages fix no
 * summation order; this layer fixes one (32 strided fmaf chains, then a
 * halving pairwise tree) so that the selection, which compares these fp32
 * values, is reproducible bit for bit. */
void orc_router_logits(const float *x, int64_t T, int64_t d, const float *Wr, int64_t E, float *logits)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t e = 0; e < E; ++e) {
            float part[32];
            for (int j = 0; j < 32; ++j)
                part[j] = 0.0f;
            for (int64_t k = 0; k < d; ++k)
                part[k % 32] = fmaf(x[t * d + k], Wr[e * d + k], part[k % 32]);
            for (int off = 16; off >= 1; off /= 2)
                for (int j = 0; j < off; ++j)
                    part[j] = part[j] + part[j + off];
            logits[t * E + e] = part[0];
        }
    }
}

/* Index of the largest value among the entries with allowed[i] != 0, the lowest index
 * winning a tie; -1 when none is allowed. A plain linear scan. */
static int argmax_allowed(const float *v, const unsigned char *allowed, int n)
{
    int best = -1;
    for (int i = 0; i < n; ++i)
        if (allowed[i] && (best < 0 || v[i] > v[best]))
            best = i;
    return best;
}

/* ---- sigmoid router with grouped top-k ----------------------------------------
 * DeepSeek-V3 style ("Router style DeepSeek-V3" row of the dashen-tech
 * "Points techniques cles" table), with the layer's grouped top-k:
 *   s_e = sigmoid(l_e), computed in fp64 and rounded to fp32;
 *   c_e = s_e + bias_e in fp32 (the bias steers selection only);
 *   experts form n_group contiguous groups of E/n_group; a group's score is the
 *   sum of its two largest c (its one c when a group has one expert);
 *   the topk_group best groups are kept (ties: lower group index);
 *   the top_k largest c among the kept experts are selected, in descending c
 *   (ties: lower expert index);
 *   w_i = s_i / sum_j s_j * routed_scale (fp64, sum in selection order), or
 *   s_i * routed_scale when renormalisation is off. */
static int select_sigmoid(const orc_cfg *cfg, const float *l, const float *bias, int32_t *ids, float *w)
{
    const int E = cfg->n_exp, G = cfg->n_group, KG = cfg->topk_group, K = cfg->top_k;
    const int gs = E / G;
    float *s = (float *)malloc(sizeof(float) * E);
    float *c = (float *)malloc(sizeof(float) * E);
    float *gscore = (float *)malloc(sizeof(float) * G);
    unsigned char *allowed = (unsigned char *)malloc(E > G ? E : G);
    unsigned char *kept = (unsigned char *)malloc(G);
    if (!s || !c || !gscore || !allowed || !kept) {
        free(s); free(c); free(gscore); free(allowed); free(kept);
        return -1;
    }
    for (int e = 0; e < E; ++e) {
        s[e] = (float)(1.0 / (1.0 + exp(-(double)l[e])));
        c[e] = s[e] + (bias ? bias[e] : 0.0f);
        if (isnan(c[e]))
            c[e] = -INFINITY;  /* a NaN score ranks below every number */
    }
    for (int g = 0; g < G; ++g) {
        const float *cg = c + g * gs;
        memset(allowed, 1, gs);
        int i1 = argmax_allowed(cg, allowed, gs);
        if (i1 < 0) {
            free(s); free(c); free(gscore); free(allowed); free(kept);
            return -1;
        }
        if (gs == 1) {
            gscore[g] = cg[i1];
        } else {
            allowed[i1] = 0;
            int i2 = argmax_allowed(cg, allowed, gs);
            gscore[g] = cg[i1] + cg[i2];
        }
    }
    memset(allowed, 1, G);
    memset(kept, 0, G);
    for (int r = 0; r < KG; ++r) {
        int g = argmax_allowed(gscore, allowed, G);
        if (g < 0)
            break;
        kept[g] = 1;
        allowed[g] = 0;
    }
    for (int e = 0; e < E; ++e)
        allowed[e] = kept[e / gs];
    for (int i = 0; i < K; ++i) {
        int e = argmax_allowed(c, allowed, E);
        ids[i] = e;
        if (e >= 0)
            allowed[e] = 0;
    }
    double sum = 0.0;
    for (int i = 0; i < K; ++i)
        sum += (double)s[ids[i]];
    for (int i = 0; i < K; ++i) {
        double p = (double)s[ids[i]];
        if (cfg->norm_topk)
            p = p / sum;
        w[i] = (float)(p * (double)cfg->routed_scale);
    }
    free(s); free(c); free(gscore); free(allowed); free(kept);
    return 0;
}

/* ---- softmax top-k router (OLMoE-shaped layer) --------------------------------
 * Top-k by logit (descending, ties: lower index); w_i = exp(l_i - m) / sum_e exp(l_e - m)
 * over all E experts in fp64 (m = max l), optionally renormalised over the k selected,
 * times routed_scale. */
static int select_softmax(const orc_cfg *cfg, const float *l, int32_t *ids, float *w)
{
    const int E = cfg->n_exp, K = cfg->top_k;
    unsigned char *allowed = (unsigned char *)malloc(E);
    float *key = (float *)malloc(sizeof(float) * E);
    if (!allowed || !key) {
        free(allowed); free(key);
        return -1;
    }
    for (int e = 0; e < E; ++e)
        key[e] = isnan(l[e]) ? -INFINITY : l[e];  /* a NaN logit ranks below every number */
    memset(allowed, 1, E);
    for (int i = 0; i < K; ++i) {
        int e = argmax_allowed(key, allowed, E);
        ids[i] = e;
        if (e >= 0)
            allowed[e] = 0;
    }
    double m = (double)l[0];
    for (int e = 1; e < E; ++e)
        if ((double)l[e] > m)
            m = (double)l[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e)
        z += exp((double)l[e] - m);
    double sel = 0.0;
    for (int i = 0; i < K; ++i)
        sel += exp((double)l[ids[i]] - m) / z;
    for (int i = 0; i < K; ++i) {
        double p = exp((double)l[ids[i]] - m) / z;
        if (cfg->norm_topk)
            p = p / sel;
        w[i] = (float)(p * (double)cfg->routed_scale);
    }
    free(allowed);
    free(key);
    return 0;
}

static int cfg_ok(const orc_cfg *cfg)
{
    if (cfg->d <= 0 || cfg->d % ORC_GROUP || cfg->ffn <= 0 || cfg->ffn % ORC_GROUP)
        return 0;
    if (cfg->n_exp <= 0 || cfg->top_k <= 0 || cfg->top_k > cfg->n_exp)
        return 0;
    if (cfg->has_shared && (cfg->shared_ffn <= 0 || cfg->shared_ffn % ORC_GROUP))
        return 0;
    if (cfg->router == ORC_ROUTER_SIGMOID_GROUPED) {
        if (cfg->n_group <= 0 || cfg->n_exp % cfg->n_group)
            return 0;
        if (cfg->topk_group <= 0 || cfg->topk_group > cfg->n_group)
            return 0;
        if (cfg->topk_group * (cfg->n_exp / cfg->n_group) < cfg->top_k)
            return 0;
    } else if (cfg->router != ORC_ROUTER_SOFTMAX) {
        return 0;
    }
    return 1;
}

int orc_router_select(const orc_cfg *cfg, const float *logits, int64_t T, const float *bias,
                      int32_t *ids, float *w)
{
    if (!cfg_ok(cfg))
        return -1;
    const int E = cfg->n_exp, K = cfg->top_k;
    for (int64_t t = 0; t < T; ++t) {
        int rc = cfg->router == ORC_ROUTER_SOFTMAX
                     ? select_softmax(cfg, logits + t * E, ids + t * K, w + t * K)
                     : select_sigmoid(cfg, logits + t * E, bias, ids + t * K, w + t * K);
        if (rc)
            return rc;
    }
    return 0;
}

int orc_router_topk(const orc_cfg *cfg, const float *x, int64_t T, const float *Wr,
                    const float *bias, int32_t *ids, float *w)
{
    if (!cfg_ok(cfg))
        return -1;
    float *logits = (float *)malloc(sizeof(float) * (size_t)(T * cfg->n_exp + 1));
    if (!logits)
        return -1;
    orc_router_logits(x, T, cfg->d, Wr, cfg->n_exp, logits);
    int rc = orc_router_select(cfg, logits, T, bias, ids, w);
    free(logits);
    return rc;
}

/* ---- bucketing ------------------------------------------------------------------
 * Counting sort of the (token, slot) pairs by expert, stable in p = t*k + i. */
int orc_bucket(const int32_t *ids, int64_t T, int k, int E, int32_t *offsets, int32_t *pairs)
{
    const int64_t P = T * k;
    for (int e = 0; e <= E; ++e)
        offsets[e] = 0;
    for (int64_t p = 0; p < P; ++p) {
        if (ids[p] < 0 || ids[p] >= E)
            return -1;
        offsets[ids[p] + 1] += 1;
    }
    for (int e = 0; e < E; ++e)
        offsets[e + 1] += offsets[e];
    int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    if (!next)
        return -1;
    for (int e = 0; e < E; ++e)
        next[e] = offsets[e];
    for (int64_t p = 0; p < P; ++p)
        pairs[next[ids[p]]++] = (int32_t)p;
    free(next);
    return 0;
}

/* ---- integer group dots ---------------------------------------------------------
 * The int8 x int4 dot of the pages' integer kernel, one int32 per group of `group`
 * columns (|dot| <= 64 * 8 * 127 = 65,024). */
static inline void group_dots_n(const uint8_t *w, const int8_t *qa, int64_t rows, int64_t cols, int group,
                                int32_t *dots)
{
    const int64_t ng = cols / group;
    int8_t q[64];
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < ng; ++g) {
            orc_unpack_int4(w + r * (cols / 2) + g * (group / 2), group / 2, q);
            int32_t acc = 0;
            for (int k = 0; k < group; ++k)
                acc += (int32_t)q[k] * (int32_t)qa[g * group + k];
            dots[r * ng + g] = acc;
        }
    }
}

int orc_group_dots_g(const uint8_t *w, const int8_t *qa, int64_t rows, int64_t cols, int group, int32_t *dots)
{
    if (!group_ok(group) || rows < 0 || cols < 0 || cols % group != 0)
        return -1;
    /* the same loop with the group size as a constant of each call */
    if (group == 64)
        group_dots_n(w, qa, rows, cols, 64, dots);
    else
        group_dots_n(w, qa, rows, cols, 32, dots);
    return 0;
}

void orc_group_dots(const uint8_t *w, const int8_t *qa, int64_t rows, int64_t cols, int32_t *dots)
{
    orc_group_dots_g(w, qa, rows, cols, ORC_GROUP, dots);
}

/* ---- one token through one SwiGLU expert ---------------------------------------
 * gate_n = sum_g s1[n][g] * sx[g] * D1[n][g], up_n likewise with W3 (fp64);
 * h_n = silu(gate_n) * up_n with silu(z) = z / (1 + exp(-z)), rounded to fp32;
 * (qh, sh) = q8(h); y_m = sum_g s2[m][g] * sh[g] * D2[m][g] (fp64), rounded to fp32. */
int orc_expert_token_g(int d, int f, int group, const orc_expert *ex, const int8_t *qx, const float *sx,
                       float *y, int8_t *qh_out, float *sh_out, float *h_out)
{
    if (!group_ok(group) || d % group || f % group)
        return -1;
    const int ngd = d / group, ngf = f / group;
    int32_t *dots = (int32_t *)malloc(sizeof(int32_t) * (size_t)(ngd > ngf ? ngd : ngf));
    float *h = (float *)malloc(sizeof(float) * (size_t)f);
    int8_t *qh = (int8_t *)malloc((size_t)f);
    float *sh = (float *)malloc(sizeof(float) * (size_t)ngf);
    if (!dots || !h || !qh || !sh) {
        free(dots); free(h); free(qh); free(sh);
        return -1;
    }
    for (int n = 0; n < f; ++n) {
        orc_group_dots_g(ex->w1 + (int64_t)n * (d / 2), qx, 1, d, group, dots);
        double gate = 0.0;
        for (int g = 0; g < ngd; ++g)
            gate += (double)ex->s1[(int64_t)n * ngd + g] * (double)sx[g] * (double)dots[g];
        orc_group_dots_g(ex->w3 + (int64_t)n * (d / 2), qx, 1, d, group, dots);
        double up = 0.0;
        for (int g = 0; g < ngd; ++g)
            up += (double)ex->s3[(int64_t)n * ngd + g] * (double)sx[g] * (double)dots[g];
        h[n] = (float)(gate / (1.0 + exp(-gate)) * up);
    }
    orc_q8_quantize_g(h, 1, f, group, qh, sh);
    for (int m = 0; m < d; ++m) {
        orc_group_dots_g(ex->w2 + (int64_t)m * (f / 2), qh, 1, f, group, dots);
        double acc = 0.0;
        for (int g = 0; g < ngf; ++g)
            acc += (double)ex->s2[(int64_t)m * ngf + g] * (double)sh[g] * (double)dots[g];
        y[m] = (float)acc;
    }
    if (qh_out)
        memcpy(qh_out, qh, (size_t)f);
    if (sh_out)
        memcpy(sh_out, sh, sizeof(float) * (size_t)ngf);
    if (h_out)
        memcpy(h_out, h, sizeof(float) * (size_t)f);
    free(dots); free(h); free(qh); free(sh);
    return 0;
}

int orc_expert_token(int d, int f, const orc_expert *ex, const int8_t *qx, const float *sx,
                     float *y, int8_t *qh_out, float *sh_out, float *h_out)
{
    return orc_expert_token_g(d, f, ORC_GROUP, ex, qx, sx, y, qh_out, sh_out, h_out);
}

/* ---- one token through one SwiGLU expert, activations kept in fp32 ------------------
 * The decode variant of the dashen-tech guide ("Analyse approfondie", step 3: one-token
 * decode runs on f32 activations) with the same int4 group-scaled weights:
 * gate_n = sum_k s1[n][k/32] * q1[n][k] * x[k] and up_n likewise (fp64, k ascending);
 * h_n = silu(gate_n) * up_n rounded to fp32; y_m = sum_j s2[m][j/32] * q2[m][j] * h_j
 * (fp64, j ascending) rounded to fp32. Nothing is quantised but the weights. */
/* group is 32 or 64: its only caller, orc_expert_token_f32_g, rejects any other size */
static double dot_row_f32(const uint8_t *wrow, const float *srow, const float *v, int K, int group, int8_t *q)
{
    orc_unpack_int4(wrow, K / 2, q);
    const int shift = group == 64 ? 6 : 5;  /* k / group */
    double acc = 0.0;
    for (int k = 0; k < K; ++k)
        acc += (double)srow[k >> shift] * (double)q[k] * (double)v[k];
    return acc;
}

int orc_expert_token_f32_g(int d, int f, int group, const orc_expert *ex, const float *x, float *y,
                           float *h_out)
{
    if (!group_ok(group) || d % group || f % group)
        return -1;
    const int ngd = d / group, ngf = f / group;
    int8_t *q = (int8_t *)malloc((size_t)(d > f ? d : f));
    float *h = (float *)malloc(sizeof(float) * (size_t)f);
    if (!q || !h) {
        free(q); free(h);
        return -1;
    }
    for (int n = 0; n < f; ++n) {
        const double gate = dot_row_f32(ex->w1 + (int64_t)n * (d / 2), ex->s1 + (int64_t)n * ngd, x, d, group, q);
        const double up = dot_row_f32(ex->w3 + (int64_t)n * (d / 2), ex->s3 + (int64_t)n * ngd, x, d, group, q);
        h[n] = (float)(gate / (1.0 + exp(-gate)) * up);
    }
    for (int m = 0; m < d; ++m)
        y[m] = (float)dot_row_f32(ex->w2 + (int64_t)m * (f / 2), ex->s2 + (int64_t)m * ngf, h, f, group, q);
    if (h_out)
        memcpy(h_out, h, sizeof(float) * (size_t)f);
    free(q); free(h);
    return 0;
}

int orc_expert_token_f32(int d, int f, const orc_expert *ex, const float *x, float *y, float *h_out)
{
    return orc_expert_token_f32_g(d, f, ORC_GROUP, ex, x, y, h_out);
}

/* ---- the layer --------------------------------------------------------------------
 * Per token t: route (or take the given ids and weights), q8 the token, run the
 * shared expert (weight 1, not scaled) and each selected expert, and combine
 * out[t] = y_shared + sum_i w[t][i] * y_i in fp64 in selection order, rounded to fp32.
 * Tokens are independent of one another. */
int orc_moe_layer_g(const orc_cfg *cfg, int group, int act_f32, const float *x, int64_t T, const float *Wr,
                    const float *bias, const orc_expert *experts, const orc_expert *shared,
                    const int32_t *ids_in, const float *w_in, int32_t *ids_out, float *w_out, float *out)
{
    if (!cfg_ok(cfg) || !group_ok(group) || T < 0 || (cfg->has_shared && !shared))
        return -1;
    if (cfg->d % group || cfg->ffn % group || (cfg->has_shared && cfg->shared_ffn % group))
        return -1;
    const int d = cfg->d, K = cfg->top_k, E = cfg->n_exp;
    const int ngd = d / group;
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T * K + 1));
    float *w = (float *)malloc(sizeof(float) * (size_t)(T * K + 1));
    int8_t *qx = (int8_t *)malloc((size_t)d);
    float *sx = (float *)malloc(sizeof(float) * (size_t)ngd);
    float *y = (float *)malloc(sizeof(float) * (size_t)d);
    double *acc = (double *)malloc(sizeof(double) * (size_t)d);
    int rc = 0;
    if (!ids || !w || !qx || !sx || !y || !acc) {
        rc = -1;
        goto done;
    }
    if (ids_in) {
        for (int64_t p = 0; p < T * K; ++p) {
            if (ids_in[p] < 0 || ids_in[p] >= E) {
                rc = -1;
                goto done;
            }
            ids[p] = ids_in[p];
            w[p] = w_in[p];
        }
    } else if (T > 0) {
        rc = orc_router_topk(cfg, x, T, Wr, bias, ids, w);
        if (rc)
            goto done;
    }
    for (int64_t t = 0; t < T; ++t) {
        const float *xt = x + t * d;
        if (!act_f32)
            orc_q8_quantize_g(xt, 1, d, group, qx, sx);
        for (int m = 0; m < d; ++m)
            acc[m] = 0.0;
        if (cfg->has_shared) {
            rc = act_f32 ? orc_expert_token_f32_g(d, cfg->shared_ffn, group, shared, xt, y, NULL)
                         : orc_expert_token_g(d, cfg->shared_ffn, group, shared, qx, sx, y, NULL, NULL, NULL);
            if (rc)
                goto done;
            for (int m = 0; m < d; ++m)
                acc[m] = (double)y[m];
        }
        for (int i = 0; i < K; ++i) {
            const orc_expert *ex = &experts[ids[t * K + i]];
            rc = act_f32 ? orc_expert_token_f32_g(d, cfg->ffn, group, ex, xt, y, NULL)
                         : orc_expert_token_g(d, cfg->ffn, group, ex, qx, sx, y, NULL, NULL, NULL);
            if (rc)
                goto done;
            for (int m = 0; m < d; ++m)
                acc[m] += (double)w[t * K + i] * (double)y[m];
        }
        for (int m = 0; m < d; ++m)
            out[t * d + m] = (float)acc[m];
    }
    if (ids_out)
        memcpy(ids_out, ids, sizeof(int32_t) * (size_t)(T * K));
    if (w_out)
        memcpy(w_out, w, sizeof(float) * (size_t)(T * K));
done:
    free(ids); free(w); free(qx); free(sx); free(y); free(acc);
    return rc;
}

int orc_moe_layer(const orc_cfg *cfg, const float *x, int64_t T, const float *Wr,
                  const float *bias, const orc_expert *experts, const orc_expert *shared,
                  const int32_t *ids_in, const float *w_in, int32_t *ids_out, float *w_out,
                  float *out)
{
    return orc_moe_layer_g(cfg, ORC_GROUP, 0, x, T, Wr, bias, experts, shared, ids_in, w_in, ids_out, w_out, out);
}

/* The same layer with every expert on fp32 activations (orc_expert_token_f32). */
int orc_moe_layer_f32(const orc_cfg *cfg, const float *x, int64_t T, const float *Wr,
                      const float *bias, const orc_expert *experts, const orc_expert *shared,
                      const int32_t *ids_in, const float *w_in, int32_t *ids_out, float *w_out,
                      float *out)
{
    return orc_moe_layer_g(cfg, ORC_GROUP, 1, x, T, Wr, bias, experts, shared, ids_in, w_in, ids_out, w_out, out);
}

/* ---- LRU cache trace -----------------------------------------------------------
 * A capacity-slot table with a use stamp per slot; the victim is the valid,
 * unpinned slot with the oldest stamp. Keys looked up since the last batch start
 * are pinned. */
int orc_lru_trace(int capacity, int64_t n_ops, const int32_t *kind, const int64_t *key,
                  int8_t *result)
{
    if (capacity <= 0)
        return -1;
    int64_t *keys = (int64_t *)calloc((size_t)capacity, sizeof(int64_t));
    int64_t *stamp = (int64_t *)calloc((size_t)capacity, sizeof(int64_t));
    unsigned char *valid = (unsigned char *)calloc((size_t)capacity, 1);
    unsigned char *pinned = (unsigned char *)calloc((size_t)capacity, 1);
    if (!keys || !stamp || !valid || !pinned) {
        free(keys); free(stamp); free(valid); free(pinned);
        return -1;
    }
    int64_t clock = 0;
    for (int64_t o = 0; o < n_ops; ++o) {
        if (kind[o] == 0) {
            memset(pinned, 0, (size_t)capacity);
            result[o] = 0;
            continue;
        }
        int found = -1;
        for (int i = 0; i < capacity; ++i)
            if (valid[i] && keys[i] == key[o])
                found = i;
        if (found >= 0) {
            stamp[found] = ++clock;
            if (kind[o] == 1)
                pinned[found] = 1;
            result[o] = 1;
            continue;
        }
        int slot = -1;
        for (int i = 0; i < capacity && slot < 0; ++i)
            if (!valid[i])
                slot = i;
        if (slot < 0) {
            for (int i = 0; i < capacity; ++i)
                if (!pinned[i] && (slot < 0 || stamp[i] < stamp[slot]))
                    slot = i;
        }
        if (slot < 0) {
            result[o] = 2;
            continue;
        }
        keys[slot] = key[o];
        valid[slot] = 1;
        stamp[slot] = ++clock;
        pinned[slot] = kind[o] == 1;
        result[o] = 0;
    }
    free(keys); free(stamp); free(valid); free(pinned);
    return 0;
}

/* The expert cache's replacement policy with a usage-pinned hot set, on abstract keys
 * (kongchang.com article, section 三级存储分层: learned-hot experts stay in the fast tier;
 * the pages give no algorithm, so this is the reading the library implements): every
 * lookup adds one use of its key; up to n_hot resident keys are hot and never evicted; a
 * key with a new use enters the hot set when there is room or when it has strictly more
 * uses than the weakest hot key (fewest uses, then least recently accessed), which leaves
 * the set but stays resident. Victims are the least recently accessed slots that are
 * neither pinned by the current lookup batch nor hot. n_hot = 0 is orc_lru_trace. Plain
 * arrays and linear scans. */
int orc_lru_hot_trace(int capacity, int n_hot, int64_t n_ops, const int32_t *kind, const int64_t *key,
                      int8_t *result)
{
    if (capacity <= 0 || n_hot < 0 || n_hot > capacity)
        return -1;
    int64_t *keys = (int64_t *)calloc((size_t)capacity, sizeof(int64_t));
    int64_t *stamp = (int64_t *)calloc((size_t)capacity, sizeof(int64_t));
    unsigned char *valid = (unsigned char *)calloc((size_t)capacity, 1);
    unsigned char *pinned = (unsigned char *)calloc((size_t)capacity, 1);
    unsigned char *hot = (unsigned char *)calloc((size_t)capacity, 1);
    int64_t *ukey = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_ops > 0 ? n_ops : 1));
    int64_t *ucnt = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_ops > 0 ? n_ops : 1));
    if (!keys || !stamp || !valid || !pinned || !hot || !ukey || !ucnt) {
        free(keys); free(stamp); free(valid); free(pinned); free(hot); free(ukey); free(ucnt);
        return -1;
    }
    int64_t n_keys = 0, clock = 0;
    for (int64_t o = 0; o < n_ops; ++o) {
        if (kind[o] == 0) {
            memset(pinned, 0, (size_t)capacity);
            result[o] = 0;
            continue;
        }
        const int lookup = kind[o] == 1;
        if (lookup) {
            int64_t u = -1;
            for (int64_t i = 0; i < n_keys; ++i)
                if (ukey[i] == key[o])
                    u = i;
            if (u < 0) {
                u = n_keys++;
                ukey[u] = key[o];
                ucnt[u] = 0;
            }
            ucnt[u] += 1;
        }
        int slot = -1;
        for (int i = 0; i < capacity; ++i)
            if (valid[i] && keys[i] == key[o])
                slot = i;
        if (slot >= 0) {
            result[o] = 1;
        } else {
            for (int i = 0; i < capacity && slot < 0; ++i)
                if (!valid[i])
                    slot = i;
            if (slot < 0) {
                for (int i = 0; i < capacity; ++i)
                    if (!pinned[i] && !hot[i] && (slot < 0 || stamp[i] < stamp[slot]))
                        slot = i;
            }
            if (slot < 0) {
                result[o] = 2;
                continue;
            }
            keys[slot] = key[o];
            valid[slot] = 1;
            hot[slot] = 0;
            pinned[slot] = 0;
            result[o] = 0;
        }
        stamp[slot] = ++clock;
        if (lookup)
            pinned[slot] = 1;
        if (!lookup || n_hot == 0 || hot[slot])
            continue;
        /* the hot-set rule, counting uses by scanning the key list */
        int n_in = 0, weakest = -1;
        int64_t wu = 0, su = 0;
        for (int i = 0; i < capacity; ++i) {
            if (!valid[i])
                continue;
            int64_t ui = 0;
            for (int64_t j = 0; j < n_keys; ++j)
                if (ukey[j] == keys[i])
                    ui = ucnt[j];
            if (i == slot)
                su = ui;
            if (!hot[i])
                continue;
            ++n_in;
            if (weakest < 0 || ui < wu || (ui == wu && stamp[i] < stamp[weakest])) {
                weakest = i;
                wu = ui;
            }
        }
        if (n_in < n_hot) {
            hot[slot] = 1;
        } else if (su > wu) {
            hot[weakest] = 0;
            hot[slot] = 1;
        }
    }
    free(keys); free(stamp); free(valid); free(pinned); free(hot); free(ukey); free(ucnt);
    return 0;
}
