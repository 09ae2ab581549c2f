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
    uint16_t *q_bf;  // optional: codes as bf16 in the tensor-core k order (bf16_pos)
    int group;       // elements per scale: 32 or 64 (corrections stay per 32 elements)
};

struct RouterArgs {
    const float *x;
    int T, d, E;
    int xt;              // token rows of x staged in shared memory per pass
    const float *Wr;
    const float *bias;   // sigmoid mode; may be null (zero bias)
    float *logits;       // [T][E]
    float *s, *c;        // [T][E] sigmoid and biased score, or null (softmax mode)
    Q8Args q8;           // q8 of x as a side job when q8.x != null
    int *err;
};

struct SelectArgs {
    const float *logits;
    const float *s, *c;  // [T][E] from k_route_logits, or null: computed from logits
    const float *bias;
    int T, E, K, n_group, topk_group, router, norm_topk;
    float routed_scale;
    int32_t *ids;
    float *w;
};

struct BucketArgs {
    const int32_t *ids;
    int T, K, E, has_shared, shared_ffn, ffn, down_blocks;
    int stage_ids;  // 1: k_bucket's shared memory also holds the T*K ids after its counters
    int32_t *offsets;
    int32_t *pairs;
    Slot *slots;
    Counters *counters;
    int *err;
};

// Decode (kernels_decode.cu).
enum { MODE_GATEUP = 0, MODE_DOWN = 1, MODE_LOGIT = 2 };
constexpr int DN_ITEM_ROWS = 32;  // rows of d per down work unit in the bucketing counters

struct DecodeArgs {
    const colibri_expert *experts;
    colibri_expert shared;
    int d, ffn, shared_ffn, T, K, has_shared, fmax;
    // routing inputs: activations [T][d], router matrix [E][d] and bias [E] (sigmoid mode;
    // may be null); unused when ids_given
    const float *x, *Wr, *bias;
    int ids_given, E, n_group, topk_group, router, norm_topk;
    float routed_scale;
    // router logits, sigmoid scores s and biased scores c [T][E], written by the logit items
    float *logits, *rs, *rc;
    int32_t *ids;       // [T][K]: given, or the selection (written by CTA 0)
    const float *w_in;  // [T][K] given weights
    float *w_out;       // [T][K] selected weights (CTA 0)
    // bucketing results (every CTA keeps its own copy in shared memory; CTA 0 writes them
    // here for inspection): bucket offsets, pair list, slots, counters
    int32_t *offsets, *pairs;
    Slot *slots;
    Counters *counters;
    // q8 of x, each CTA's share quantised by its epilogue warps: plain codes (for
    // inspection), codes in even/odd word order, scales, corrections 8 * sum(codes) per
    // 32-group (read by every CTA once the routing counter is complete)
    int8_t *qx, *xq_eo;
    float *sx;
    int *xc;
    // q8(h) (row = pair; the shared expert's rows follow the T*K routed pairs; scales and
    // corrections hgs to a row), written by the gate/up items and read by the down items
    int8_t *hq, *hq_eo;
    float *hs;
    int *hc;
    float *y;    // down outputs [pairs][d]
    float *out;  // layer output [T][d]
    // zeroed per call: the work-claim counter, the routing counter (logit tasks (expert,
    // token) and q8 groups of x done), finished rows of h per slot, finished rows of y per
    // row block of d
    int *claim, *route_done, *done_gu, *done_rb;
    int *err;
    int max_slots;  // the shared expert + min(E, T*K) routed slots
    // set by launch_decode: ring stages, h buffers, partial-sum buffers (= epilogue warps),
    // tokens per chunk, groups per h row; logit items: experts and tokens per item, K
    // columns per stage, stages per item, items (0 with the ids given); warps that select
    // at once
    int ring, nh, nbuf, tch, hgs;
    int lg_ne, lg_tb, lg_kc, lg_nck, n_logit, sel_warps;
    // quantisation group (32 or 64); with 64, the gate/up items' fp32 h rows and one
    // counter per (row of h, 64-group): the item that completes a pair quantises it
    int group;
    float *hf;
    int *hpair;
};

// One persistent launch for a decode step: router logits, expert selection (unless
// ids_given) and bucketing, then gate/up, down and the combine.
cudaError_t launch_decode(DecodeArgs a, cudaStream_t s);

// Several layers in one persistent launch: layer l + 1 reads layer l's output as its
// activations. The layers share shapes, workspace and launch geometry; their control
// words alternate between two areas (CTA 0 clears the one the next layer takes), and
// the CTAs meet on a grid barrier (a counter) between layers.
constexpr int STACK_MAX = 16;
struct DecodeStack {
    DecodeArgs layer[STACK_MAX];
    int L;
    int *bar;         // grid barrier: CTAs arrived, over all layer boundaries
    int *sync_area[2];
    int sync_words;   // ints of one control-word area
};
cudaError_t launch_decode_stack(DecodeStack &p, cudaStream_t s);

// Scales (and corrections) a row of q8(h) holds on the decode path: fmax/32 rounded up to
// 16 bytes.
int decode_hgs(int fmax);

// Prefill grouped GEMMs on tcgen05 (kernels_gemm.cu).
struct GemmArgs {
    const colibri_expert *experts;
    colibri_expert shared;
    int d, ffn, shared_ffn, T, K, has_shared, fmax;
    const Slot *slots;
    const Counters *counters;
    const int32_t *pairs;
    // activations: codes as bf16 in the tensor-core k order, and their group scales; x
    // for gate/up (row = token), q8(h) for down (row = pair)
    const uint16_t *abf;
    const float *as;
    long act_stride;   // elements between activation rows of abf
    int act_groups;    // groups between activation rows of as
    uint16_t *hbf;     // gate/up output: q8(h) codes as bf16 [pairs_total][fmax]
    float *hs;         // gate/up output: their scales [pairs_total][fmax/32]
    float *y;          // down output [pairs_total][d]
    int group;         // quantisation group: 32 or 64 (one scale per group of 32-column tiles)
    int *err;
};

cudaError_t launch_gemm(int mode, const GemmArgs &a, cudaStream_t s);

// tcgen05 test export (kernels_gemm.cu)
__global__ void k_debug_umma(const int8_t *a, const int8_t *b, int n, int k, int32_t *d, int *err);
size_t debug_umma_smem(int n, int k);

// Decode on fp32 activations (kernels_f32act.cu).
struct F32Args {
    const colibri_expert *experts;  // device table [E]
    colibri_expert shared;          // members are device pointers (unused when !has_shared)
    const int32_t *ids;             // [T][K]
    const float *x;                 // [T][d]
    float *h;                       // [T*K + T][fmax]: pairs, then the shared expert's rows
    float *y;                       // [T*K + T][d]
    int T, K, E, d, ffn, shared_ffn, has_shared, fmax;
    int gsh;  // 1 for 64-element groups (the scale of 32-column tile g is group g >> gsh)
    int *err;
};
__global__ void k_f32_gateup(F32Args a);
__global__ void k_f32_down(F32Args a);
size_t f32_smem_gateup(int d);
size_t f32_smem_down(int fmax);

struct CombineArgs {
    const float *y;
    const float *w;
    int T, K, d, has_shared;
    float *out;
};


__global__ void k_q8(Q8Args a);
__global__ void k_route_logits(RouterArgs a);
__global__ void k_route_logits_tiled(RouterArgs a);
constexpr size_t ROUTE_TILED_SMEM = 2 * (16 + 32) * 256 * 4;  // two stages of a 16-token x 32-expert tile, 256 columns
size_t bucket_smem_bytes(int E, int nthreads);
__global__ void k_router_select(SelectArgs a);
__global__ void k_bucket(BucketArgs a);
__global__ void k_combine(CombineArgs a);
__global__ void k_debug_dots(const uint8_t *w, const int8_t *qa, int rows, int cols, int32_t *dots);


}  // namespace clb
