// Kernel argument blocks and launch declarations (device side of libcolibri.so).
#pragma once

#include "common.cuh"

namespace clb {

struct Q8Args {
    const float *x;
    long rows;
    int cols;
    int8_t *q;
    float *scale;
    int8_t *q_eo;  // optional: codes in even/odd word order
    int *corr;     // optional: 8 * sum(codes) per group
    int *err;      // optional: cleared by block 0
};

struct RouterArgs {
    const float *x;
    int T, d, E;
    const float *Wr;
    float *logits;
    int *err;
};

struct SelectArgs {
    const float *logits;
    const float *bias;
    int T, E, K, n_group, topk_group, router, norm_topk;
    float routed_scale;
    int32_t *ids;
    float *w;
};

struct BucketArgs {
    const int32_t *ids;
    int T, K, E, has_shared, shared_ffn, ffn, down_blocks;
    int32_t *offsets;
    int32_t *pairs;
    Slot *slots;
    Counters *counters;
    int *err;
};

// Decode gate/up: one CTA per (slot, 32-row block of f). Activations: even/odd codes,
// scales and corrections of x per token.
struct GateUpArgs {
    const colibri_expert *experts;
    colibri_expert shared;
    int d, ffn, shared_ffn, T, K, has_shared, fmax;
    const Slot *slots;
    const Counters *counters;
    const int32_t *pairs;
    const int8_t *xq_eo;
    const float *xs;
    const int *xc;
    int8_t *hq;     // [pairs_total][fmax] plain codes
    int8_t *hq_eo;  // [pairs_total][fmax] even/odd codes
    float *hs;      // [pairs_total][fmax/32]
    int *hc;        // [pairs_total][fmax/32]
};

// Decode down: one CTA per (slot, 64-row block of d).
struct DownArgs {
    const colibri_expert *experts;
    colibri_expert shared;
    int d, ffn, shared_ffn, T, K, has_shared, fmax;
    const Slot *slots;
    const Counters *counters;
    const int32_t *pairs;
    const int8_t *hq_eo;
    const float *hs;
    const int *hc;
    float *y;  // [pairs_total][d]
};

struct CombineArgs {
    const float *y;
    const float *w;
    int T, K, d, has_shared;
    float *out;
};

constexpr int GU_ROWS = 32;     // rows of f per gate/up item (one h group)
constexpr int GU_WARPS = 8;
constexpr int DN_ROWS = 64;     // rows of d per down item
constexpr int DN_WARPS = 8;
constexpr int TOK_CHUNK = 32;   // tokens held in shared memory per gate/up pass

__global__ void k_q8(Q8Args a);
__global__ void k_router_logits(RouterArgs a);
__global__ void k_router_select(SelectArgs a);
__global__ void k_bucket(BucketArgs a);
__global__ void k_combine(CombineArgs a);
__global__ void k_debug_dots(const uint8_t *w, const int8_t *qa, int rows, int cols, int32_t *dots);

cudaError_t launch_gateup(const GateUpArgs &a, int grid, cudaStream_t s);
cudaError_t launch_down(const DownArgs &a, int grid, cudaStream_t s);

}  // namespace clb
