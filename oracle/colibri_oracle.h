/*
 * colibri_oracle.h -- plain, slow CPU oracle for one routed MoE FFN layer.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package's smoke check and the
 * CPU-baseline leg of the benchmark may load this library. The CUDA library
 * shares no code, header, table or helper with it, and neither includes the
 * other.
 *
 * What it computes (the method of the Colibri expert-streaming MoE engine, as
 * described on the pages "Guide Complet de Colibri" (dashen-tech.com), the
 * kongchang.com article on Colibri, and the aifrontierpost.com Colibri
 * tutorial):
 *   - int8 activation codes per 32-element group (absmax scaling), the
 *     activation side of the "int8 x packed int4" integer dot kernel
 *     ("Points techniques cles" table, integer dot-product row, dashen-tech);
 *   - int4 expert weights with one fp32 scale per 32-element group (the
 *     group-scaled int4 container, "Step 3 -- Get a model", aifrontierpost;
 *     the pages' container uses 64-element groups, this layer uses 32);
 *   - a DeepSeek-V3-style sigmoid router with a selection bias, grouped top-k
 *     and a shared expert ("Router style DeepSeek-V3" row, same table), or a
 *     softmax top-k router for the OLMoE-shaped layer;
 *   - a SwiGLU expert MLP (gate/up, SiLU, down) on the integer group dots;
 *   - a weighted combine of the selected experts plus the shared expert;
 *   - the LRU hit/miss sequence of a small expert cache ("Streaming
 *     d'experts" bullet, dashen-tech; three-tier storage section, kongchang).
 *
 * Precision: integer work is exact (int32 group dots); floating point is
 * fp64 except where a step is defined on fp32 values (the q8 quantiser, the
 * router logits and the selection compares), which the comments state.
 * Every function is single-threaded and does no blocking, fusion or
 * reordering beyond what its comment states.
 *
 * All matrices are row-major. Weight matrices are [out][in]: row n holds the
 * in-dimension contiguously as packed nibbles, byte j of a row holding element
 * 2j in its low nibble and element 2j+1 in its high nibble, each nibble the
 * offset-binary code q+8 of q in [-8, 7]. Scales are [out][in/32] fp32.
 */
#ifndef COLIBRI_ORACLE_H
#define COLIBRI_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_GROUP 32

enum { ORC_ROUTER_SIGMOID_GROUPED = 0, ORC_ROUTER_SOFTMAX = 1 };

typedef struct {
    int d;            /* hidden size */
    int ffn;          /* routed expert intermediate size */
    int n_exp;        /* routed experts E */
    int top_k;        /* experts per token k */
    int n_group;      /* expert groups (sigmoid router) */
    int topk_group;   /* groups kept (sigmoid router) */
    int has_shared;   /* 1: one shared expert applied to every token */
    int shared_ffn;   /* shared expert intermediate size */
    int router;       /* ORC_ROUTER_* */
    int norm_topk;    /* 1: renormalise the k selected weights to sum 1 */
    float routed_scale; /* multiplies the routed weights */
} orc_cfg;

typedef struct {
    const uint8_t *w1, *w3, *w2; /* gate [f][d/2], up [f][d/2], down [d][f/2] */
    const float *s1, *s3, *s2;   /* [f][d/32], [f][d/32], [d][f/32] */
} orc_expert;

/* Offset-binary nibbles -> signed codes: q[2j] = lo(p[j]) - 8, q[2j+1] = hi(p[j]) - 8. */
void orc_unpack_int4(const uint8_t *packed, int64_t nbytes, int8_t *q);

/* Per row, per 32-group: amax = max|x|, d = amax/127 (fp32), q = clamp(roundf(x/d), -127, 127);
 * amax == 0 gives d = 0 and all-zero codes. cols % 32 == 0. Returns 0, or -1 on bad sizes. */
int orc_q8_quantize(const float *x, int64_t rows, int64_t cols, int8_t *q, float *scale);
/* The same per `group` (32 or 64) elements; scale [rows][cols/group]. */
int orc_q8_quantize_g(const float *x, int64_t rows, int64_t cols, int group, int8_t *q, float *scale);

/* Router logits l[t][e] = x[t] . Wr[e] in fp32 in one fixed order: partial sum j in [0,32)
 * accumulates x[k]*Wr[e][k] with fmaf over k = j, j+32, ... ascending; then, for
 * off = 16, 8, 4, 2, 1, partial j <- partial j + partial (j + off) for j < off; l = partial 0. */
void orc_router_logits(const float *x, int64_t T, int64_t d, const float *Wr, int64_t E, float *logits);

/* Selection and weights from logits (see the .c file for the exact steps). ids [T][k] in
 * selection order, w [T][k]. bias may be NULL (zero). Returns 0, or -1 on a bad config. */
int orc_router_select(const orc_cfg *cfg, const float *logits, int64_t T, const float *bias,
                      int32_t *ids, float *w);

/* orc_router_logits followed by orc_router_select. */
int orc_router_topk(const orc_cfg *cfg, const float *x, int64_t T, const float *Wr,
                    const float *bias, int32_t *ids, float *w);

/* Stable counting sort of the T*k (token, slot) pairs by expert: offsets [E+1] is the
 * exclusive scan of the per-expert counts, pairs [T*k] holds p = t*k + i, sorted by
 * (expert, p). Returns 0, or -1 when an id is out of range. */
int orc_bucket(const int32_t *ids, int64_t T, int k, int E, int32_t *offsets, int32_t *pairs);

/* dots[r][g] = sum over the 32 k in group g of unpack(w)[r][k] * qa[k] (int32). */
void orc_group_dots(const uint8_t *w, const int8_t *qa, int64_t rows, int64_t cols, int32_t *dots);
/* The same per `group` (32 or 64) columns; dots [rows][cols/group]. Returns 0, or -1
 * (dots untouched) for another group size or cols not a multiple of it. */
int orc_group_dots_g(const uint8_t *w, const int8_t *qa, int64_t rows, int64_t cols, int group, int32_t *dots);

/* One token through one expert of intermediate size f: gate/up group dots, SwiGLU,
 * q8 of h, down group dots. y [d] fp32; qh [f] and sh [f/32] receive h's codes and h_out
 * [f] the fp32 h they quantise (each may be NULL). Returns 0, or -1 on allocation
 * failure. */
int orc_expert_token(int d, int f, const orc_expert *ex, const int8_t *qx, const float *sx,
                     float *y, int8_t *qh, float *sh, float *h_out);
/* The same with quantisation groups of `group` (32 or 64) elements, for weights and
 * activations alike: the expert's scales are [f][d/group], [f][d/group], [d][f/group],
 * sx [d/group], sh [f/group]. Returns -1 also for a group size that does not divide d, f. */
int orc_expert_token_g(int d, int f, int group, const orc_expert *ex, const int8_t *qx, const float *sx,
                       float *y, int8_t *qh, float *sh, float *h_out);

/* One token through one expert on fp32 activations (the f32 decode variant): gate and
 * up are fp64 sums over k of scale * int4 code * x[k], h = silu(gate) * up rounded to
 * fp32, y = the same sums of W2 against h. x [d], y [d]; h_out [f] may be NULL.
 * Returns 0, or -1 on allocation failure. */
int orc_expert_token_f32(int d, int f, const orc_expert *ex, const float *x, float *y, float *h_out);
int orc_expert_token_f32_g(int d, int f, int group, const orc_expert *ex, const float *x, float *y,
                           float *h_out);

/* The whole layer for T tokens. experts [E] (routed), shared (NULL when !has_shared).
 * ids_in/w_in: when ids_in != NULL the router is skipped and ids_in/w_in [T][k] are used.
 * ids_out/w_out (may be NULL) receive the ids and weights used. out [T][d].
 * Returns 0, or -1 on bad input. */
int orc_moe_layer(const orc_cfg *cfg, const float *x, int64_t T, const float *Wr,
                  const float *bias, const orc_expert *experts, const orc_expert *shared,
                  const int32_t *ids_in, const float *w_in, int32_t *ids_out, float *w_out,
                  float *out);
/* The layer with quantisation groups of `group` (32 or 64) elements, on int8 (act_f32 = 0)
 * or fp32 (act_f32 = 1) activations. orc_moe_layer is (group 32, int8). */
int orc_moe_layer_g(const orc_cfg *cfg, int group, int act_f32, const float *x, int64_t T, const float *Wr,
                    const float *bias, const orc_expert *experts, const orc_expert *shared,
                    const int32_t *ids_in, const float *w_in, int32_t *ids_out, float *w_out, float *out);

/* orc_moe_layer with every expert on fp32 activations (orc_expert_token_f32). */
int orc_moe_layer_f32(const orc_cfg *cfg, const float *x, int64_t T, const float *Wr,
                      const float *bias, const orc_expert *experts, const orc_expert *shared,
                      const int32_t *ids_in, const float *w_in, int32_t *ids_out, float *w_out,
                      float *out);

/* LRU cache trace. ops: kind 0 = start of a lookup batch (unpins every key),
 * kind 1 = lookup key (demand), kind 2 = stage key (prefetch). result per op:
 *   kind 0: 0;
 *   kind 1: 1 hit (resident), 0 miss (inserted, evicting the least recently used
 *           unpinned key when full), 2 no unpinned key to evict; the key is then pinned;
 *   kind 2: 1 already resident, 0 inserted (same eviction rule), 2 no room (skipped).
 * Every lookup or stage of a key, hit or not, makes it the most recently used. */
int orc_lru_trace(int capacity, int64_t n_ops, const int32_t *kind, const int64_t *key,
                  int8_t *result);
int orc_lru_hot_trace(int capacity, int n_hot, int64_t n_ops, const int32_t *kind, const int64_t *key,
                      int8_t *result);

#ifdef __cplusplus
}
#endif
#endif
