/*
 * colibri.h -- C ABI of libcolibri.so: one routed Mixture-of-Experts FFN layer on a
 * B300 GPU (sm_103a), with int4 group-scaled expert weights, int8 activations and a
 * small HBM expert cache fed from pinned host memory.
 *
 * The layer is the hot path of the Colibri expert-streaming MoE engine described on
 * the pages "Guide Complet de Colibri" (dashen-tech.com), "Colibri纯C引擎爆火"
 * (kongchang.com) and "Run a 744B-parameter model on your own machine"
 * (aifrontierpost.com). Each entry point below cites the passage that defines its
 * operation.
 *
 * Conventions shared by every entry point:
 *   - Pointers named "device" are CUDA device pointers; "host" pointers are ordinary
 *     host memory. The caller allocates and owns every buffer passed in (device
 *     memory, pinned host memory, streams); the library never frees caller memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Compute entry points only enqueue work on it and return without synchronising,
 *     except colibri_moe_layer_host, which waits for its stream.
 *   - Activations are row-major. A packed int4 weight matrix W [R][K] (R = out, K = in,
 *     both multiples of 32) is stored in row blocks of 32 rows, group-major inside a
 *     block: the 16 bytes of group g (columns 32g..32g+31) of row r are at byte
 *         ((r / 32) * (K / 32) + g) * 512 + (r % 32) * 16,
 *     and byte j of them holds column 32g+2j in its low nibble and 32g+2j+1 in its high
 *     nibble, each nibble the offset-binary code q+8 of q in [-8, 7]. Its fp32 scales,
 *     one per row and group, are stored alike: S[r][g] at float
 *         ((r / 32) * (K / 32) + g) * 32 + r % 32.
 *     A warp reading group g of a row block then loads 512 contiguous bytes. The layout
 *     is this library's choice: the pages fix the group scaling, not the byte order.
 *   - Every function returns COLIBRI_OK (0) or a negative COLIBRI_E_* code. Argument
 *     errors are detected on the host before anything is enqueued. Launch errors are
 *     returned as COLIBRI_E_CUDA. Errors found on the device (an expert id out of
 *     range, a wait that ran out) set a flag in the workspace that
 *     colibri_workspace_status reports; the kernels then skip the bad work and return.
 */
#ifndef COLIBRI_H
#define COLIBRI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define COLIBRI_OK 0
#define COLIBRI_E_INVAL (-1)   /* bad argument or configuration */
#define COLIBRI_E_CUDA (-2)    /* a CUDA runtime call or launch failed */
#define COLIBRI_E_NOMEM (-3)   /* workspace or cache pool too small */
#define COLIBRI_E_TIMEOUT (-4) /* a bounded wait ran out */
#define COLIBRI_E_MISS (-5)    /* strict cache lookup found an expert not resident */
#define COLIBRI_E_STAGE (-6)   /* staging an expert into the cache failed */
#define COLIBRI_E_DEVICE (-7)  /* a kernel reported bad input through the error flag */

#define COLIBRI_GROUP 32   /* the default quantisation group: elements per scale */
#define COLIBRI_GROUP64 64 /* the 64-element groups of the pages' int4 containers */

enum { COLIBRI_ROUTER_SIGMOID_GROUPED = 0, COLIBRI_ROUTER_SOFTMAX = 1 };

/* Shape and routing of one layer.
 *   d            hidden size (multiple of 32)
 *   ffn          routed expert intermediate size (multiple of 32)
 *   n_exp        routed experts E (<= 1024), top_k experts per token (<= 32)
 *   n_group, topk_group   sigmoid router: E/n_group contiguous experts per group,
 *                topk_group groups kept
 *   has_shared, shared_ffn   one shared expert applied to every token with weight 1
 *   router       COLIBRI_ROUTER_*
 *   norm_topk    1: the k selected weights are renormalised to sum 1 before scaling
 *   routed_scale multiplies the routed weights
 *   group        elements per scale, COLIBRI_GROUP (32) or COLIBRI_GROUP64 (64): of the
 *                expert weights (one fp32 scale per row and group of columns) and of the
 *                q8 activations x and h (one scale per row and group); d, ffn and
 *                shared_ffn must be multiples of it. The int4 container of the
 *                aifrontierpost tutorial ("Step 3 -- Get a model") uses 64. */
typedef struct {
    int d, ffn, n_exp, top_k, n_group, topk_group, has_shared, shared_ffn, router, norm_topk;
    float routed_scale;
    int group;
} colibri_layer_cfg;

/* One expert's tensors (device pointers, 16-byte aligned), in the stored layout above:
 * gate w1 [f][d], up w3 [f][d], down w2 [d][f] packed int4; scales s1 [f][d/g],
 * s3 [f][d/g], s2 [d][f/g] fp32 for the layer's group g. Group-scaled int4 container:
 * aifrontierpost tutorial, "Step 3 -- Get a model". With g = 64 the nibbles are stored
 * exactly as for 32 (a 64-group is two consecutive 32-column tiles of a row block) and the
 * scales S[r][g] at float ((r / 32) * (K / 64) + g) * 32 + r % 32. */
typedef struct {
    const uint8_t *w1, *w3, *w2;
    const float *s1, *s3, *s2;
} colibri_expert;

/* Byte offsets of the six parts inside one contiguous expert blob (w1|w3|w2|s1|s3|s2,
 * each 256-byte aligned) and the blob's size. The cache stages whole blobs. */
typedef struct {
    size_t w1, w3, w2, s1, s3, s2, nbytes;
} colibri_blob_layout;

/* Host only. Fills *out for an expert of hidden size d and intermediate size f.
 * The GLM-5.2-shaped expert (d=6144, f=2048) has 18,874,368 bytes of nibbles, the
 * "~19 MB" routed expert of the kongchang.com article (section 核心思路), and
 * 23,592,960 bytes with its scales. Returns COLIBRI_E_INVAL unless d, f are positive
 * multiples of 32. */
int colibri_blob_layout_for(int d, int f, colibri_blob_layout *out);
/* The same for experts with `group`-element scale groups (32 or 64; d, f multiples of
 * it): the nibbles are the same, the scale parts are d*f/group floats each. */
int colibri_blob_layout_for_g(int d, int f, int group, colibri_blob_layout *out);

/* Host only. A static string naming a status code. */
const char *colibri_strerror(int status);

/* q8 activation quantiser (the int8 side of the int8 x packed-int4 dot kernel:
 * dashen-tech guide, table "Points techniques cles", integer dot-product row).
 * Per row and per 32 consecutive columns: d = amax/127 in fp32, q = clamp(roundf(x/d),
 * -127, 127), rounding halves away from zero; an all-zero group gets d = 0 and zero
 * codes.
 *   x      device fp32 [rows][cols], cols % 32 == 0
 *   q      device int8 [rows][cols] (out)
 *   scale  device fp32 [rows][cols/32] (out)
 * rows == 0 is a no-op. */
int colibri_q8_quantize(const float *x, int rows, int cols, int8_t *q, float *scale, void *stream);
/* The same quantiser per `group` (32 or 64) consecutive columns: scale [rows][cols/group],
 * cols % group == 0 (64: the 64-element groups of the aifrontierpost tutorial, "Step 3"). */
int colibri_q8_quantize_g(const float *x, int rows, int cols, int group, int8_t *q, float *scale,
                          void *stream);

/* Router: logits, selection and weights for T tokens (DeepSeek-V3-style sigmoid router
 * with a selection bias: dashen-tech guide, table "Points techniques cles", row "Router
 * style DeepSeek-V3"; softmax top-k for OLMoE-shaped layers).
 *   logits l[t][e] = x[t] . Wr[e] in fp32 with a fixed summation order: 32 strided
 *   fmaf chains (chain j takes k = j, j+32, ... ascending) joined by a halving pairwise
 *   tree, so that the selection is reproducible bit for bit.
 *   Sigmoid mode: s = fp32(sigmoid(l)) evaluated in fp64, c = s + bias (fp32); group
 *   score = sum of the two largest c of each of n_group contiguous groups; keep the
 *   topk_group best groups; select the top_k largest c inside them in descending order
 *   (ties: lower index, for groups and experts); w_i = s_i / sum_j s_j * routed_scale
 *   (or s_i * routed_scale when norm_topk = 0).
 *   Softmax mode: top_k largest logits (ties: lower index); w_i = softmax over all E
 *   logits at i (renormalised over the k when norm_topk = 1) * routed_scale.
 *   x       device fp32 [T][d], Wr device fp32 [E][d], both 16-byte aligned
 *   bias    device fp32 [E] or NULL (zero); ignored in softmax mode
 *   logits  device fp32 [T][E] (out; also the kernel's scratch)
 *   ids     device int32 [T][top_k] (out), w device fp32 [T][top_k] (out)
 * T == 0 is a no-op. */
int colibri_router_topk(const colibri_layer_cfg *cfg, const float *x, int T, const float *Wr,
                        const float *bias, float *logits, int32_t *ids, float *w, void *stream);

/* Bytes of device workspace colibri_moe_layer needs for up to T_max tokens
 * (0 on a bad configuration). */
size_t colibri_moe_workspace_bytes(const colibri_layer_cfg *cfg, int T_max);

/* One routed MoE FFN layer for T tokens (the expert MLP the pages run on the integer
 * dot kernel: dashen-tech guide, "Analyse approfondie" step 3; shared experts resident
 * next to the routed ones: kongchang.com article, section 核心思路).
 *   q8(x) -> router (unless ids_given) -> bucketing of (token, slot) pairs by expert ->
 *   per expert: gate = W1 q8(x), up = W3 q8(x) as int32 group dots times the two
 *   groups' scales; h = silu(gate) * up; down y = W2 q8(h) likewise ->
 *   out[t] = y_shared[t] + sum_i w[t][i] * y_{ids[t][i]}[t] in slot order.
 *   T <= 32 (decode) runs one persistent kernel: q8(x) and the router logits spread over
 *   every CTA, then each CTA selects and buckets for itself and runs its share of
 *   gate/up, down and the combine. Larger T (prefill) runs q8, router logits, selection,
 *   bucketing, the two grouped GEMMs on tcgen05 and the combine.
 *   x        device fp32 [T][d]
 *   Wr, bias as for colibri_router_topk (unused when ids_given)
 *   experts  device array of E colibri_expert (only the selected ids are read)
 *   shared   host pointer to one colibri_expert of intermediate size shared_ffn whose
 *            members are device pointers; NULL when cfg->has_shared == 0
 *   ids, w   device [T][top_k]: outputs of the router, or inputs when ids_given != 0
 *            (then the k ids of a token must be distinct and in [0, E); others set the
 *            device error flag)
 *   out      device fp32 [T][d]
 *   workspace  device, >= colibri_moe_workspace_bytes(cfg, T) bytes, 256-byte aligned;
 *            owned by the caller, must not be shared by calls that overlap on the GPU
 * T == 0 is a no-op. */
int colibri_moe_layer(const colibri_layer_cfg *cfg, const float *x, int T, const float *Wr,
                      const float *bias, const colibri_expert *experts,
                      const colibri_expert *shared, int32_t *ids, float *w, int ids_given,
                      float *out, void *workspace, size_t ws_bytes, void *stream);

/* Several decode layers in one launch (the next layer's router and shared expert are
 * sent towards L2 while the current layer drains, in the spirit of the dashen-tech
 * guide's section "Router-Lookahead prefetch"). Layer l computes colibri_moe_layer on
 * its own weights and activations: layers[l].x when given, else the previous layer's
 * out (the call's x for layer 0). The results equal n_layers sequential
 * colibri_moe_layer calls bit for bit. The CTAs meet on a grid barrier between layers.
 * Every layer shares cfg, T and ids_given. (A chain of these layers alone, out into x,
 * is not a model: each SwiGLU layer about squares the activations' magnitude, so long
 * chains overflow; a model normalises between layers, outside this library.)
 *   1 <= n_layers <= COLIBRI_STACK_MAX, 0 <= T <= 32 (decode only)
 *   layers[l]  per layer: x (device fp32 [T][d], 16-byte aligned, or NULL), Wr, bias (as
 *              colibri_moe_layer; unused when ids_given), experts, shared (host pointer,
 *              as colibri_moe_layer), ids and w (device [T][top_k], outputs or inputs as
 *              in colibri_moe_layer), out (device fp32 [T][d], 16-byte aligned). layers[]
 *              itself is host memory, read during the call. out of layer l must differ
 *              from its input; a chained layer may write the buffer of layer l - 2 (two
 *              buffers in turn suffice).
 *   workspace  device, >= colibri_moe_stack_workspace_bytes(cfg, T) bytes, 256-byte
 *              aligned, owned by the caller; the error flag is read as for
 *              colibri_moe_layer (colibri_workspace_status).
 * COLIBRI_E_INVAL for a bad argument, COLIBRI_E_NOMEM for a short workspace; T == 0 is a
 * no-op. */
#define COLIBRI_STACK_MAX 16
typedef struct {
    const float *x;
    const float *Wr;
    const float *bias;
    const colibri_expert *experts;
    const colibri_expert *shared;
    int32_t *ids;
    float *w;
    float *out;
} colibri_stack_layer;

/* Bytes of device workspace colibri_moe_stack_decode needs for up to T_max tokens (0 on
 * a bad configuration or T_max > 32). */
size_t colibri_moe_stack_workspace_bytes(const colibri_layer_cfg *cfg, int T_max);

int colibri_moe_stack_decode(const colibri_layer_cfg *cfg, const float *x, int T, int n_layers,
                             const colibri_stack_layer *layers, int ids_given, void *workspace,
                             size_t ws_bytes, void *stream);

/* colibri_moe_layer without a caller-supplied workspace. The pages have no counterpart
 * to this entry point: it exists for callers that cannot allocate device memory when
 * they run the layer (a host runtime that owns all device memory through its own pool
 * and forbids other allocations after start-up, a plugin handed only its input and
 * output buffers, a latency-critical loop that cannot afford cudaMalloc's implicit
 * device synchronisation).
 *   The workspace is a fixed array of COLIBRI_NOALLOC_SCRATCH_BYTES (16 MiB) that the
 *   library holds in the memory of every device it is loaded on, until the process
 *   exits. The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 *   library routine. The first call made in a device's context looks up the array's
 *   device address there (cudaGetSymbolAddress, which may load the library's module);
 *   make that first call before any stream capture. The address is kept per device
 *   with the id of the context it belongs to: after a cudaDeviceReset (or the primary
 *   context released and created again) the next call looks it up afresh, so a call
 *   never uses an address of a destroyed context.
 *   Arguments, layouts and results are those of colibri_moe_layer. Returns
 *   COLIBRI_E_NOMEM when colibri_moe_workspace_bytes(cfg, T) exceeds the array (the
 *   GLM-5.2-shaped layer fits up to T = 32), COLIBRI_E_INVAL on a bad configuration.
 *   Every call on a device shares the one array and leaves its contents behind for
 *   the next call; each call rewrites what it reads (the layer's host code clears the
 *   error flag and the kernels' sync counters with a memset before its first kernel).
 *   Calls whose work overlaps on the GPU (other streams, other host threads) race on
 *   the array and corrupt each other's results: serialise them.
 *   Device-side errors (an id out of range) are skipped by the kernels as in
 *   colibri_moe_layer; this variant offers no reader for the flag. */
#define COLIBRI_NOALLOC_SCRATCH_BYTES (16u << 20)
int colibri_moe_layer_noalloc(const colibri_layer_cfg *cfg, const float *x, int T, const float *Wr,
                              const float *bias, const colibri_expert *experts,
                              const colibri_expert *shared, int32_t *ids, float *w, int ids_given,
                              float *out, void *stream);

/* The layer on fp32 activations, for decode (T <= 32): the token is not quantised, as in
 * the pages' one-token decode ("Analyse approfondie", step 3 of the dashen-tech guide),
 * against the same int4 group-scaled weights. For each pair (token, selected or shared
 * expert): gate_n = sum_g s1[n][g] * sum_k q1[n][k] x[k] and up_n likewise in fp32, h =
 * silu(gate) * up in fp32, y_m = sum_g s2[m][g] * sum_j q2[m][j] h[j]; out as in
 * colibri_moe_layer. Routing is colibri_router_topk's. Weights are read once per pair.
 *   Arguments, layouts and ownership as for colibri_moe_layer, except the workspace:
 *   >= colibri_moe_f32_workspace_bytes(cfg, T) bytes, 256-byte aligned (0 from that
 *   function for a bad configuration or T_max > 32). colibri_workspace_status reads its
 *   error flag. A given id outside [0, E) sets the flag and its pair contributes nothing;
 *   a repeated id is computed twice. Returns COLIBRI_E_INVAL for T > 32. T == 0 is a no-op. */
size_t colibri_moe_f32_workspace_bytes(const colibri_layer_cfg *cfg, int T_max);
int colibri_moe_layer_f32(const colibri_layer_cfg *cfg, const float *x, int T, const float *Wr,
                          const float *bias, const colibri_expert *experts,
                          const colibri_expert *shared, int32_t *ids, float *w, int ids_given,
                          float *out, void *workspace, size_t ws_bytes, void *stream);

/* colibri_moe_layer on HOST buffers, as one blocking call: the layer computed on the
 * host side of the hybrid CPU/GPU engine of the pages ("Streaming d'experts", "Guide
 * Complet de Colibri") hands one step's activations to the GPU and takes the output back.
 * On `stream` it copies x (and ids, w when ids_given) from host memory into a region at
 * the end of the workspace, runs colibri_moe_layer on those device copies, copies out
 * (and ids, w when routed here and the pointers are non-NULL) and the device error flag
 * (into a page-locked word of the calling thread, allocated on its first call) back, and
 * waits for the stream. Host buffers may be pinned (cudaHostAlloc or
 * cudaHostRegister: the copies then run at PCIe speed without staging) or pageable
 * (correct, slower).
 *   x         host fp32 [T][d]
 *   Wr, bias, experts, shared   device, as for colibri_moe_layer
 *   ids, w    host [T][top_k]: inputs when ids_given (both required), else outputs,
 *             each optional (NULL: not copied back)
 *   out       host fp32 [T][d]
 *   workspace device, >= colibri_moe_host_workspace_bytes(cfg, T) bytes, 256-byte
 *             aligned; owned by the caller; its first colibri_moe_workspace_bytes(cfg, T)
 *             bytes are the layer's workspace
 * Returns COLIBRI_OK when out holds the result; COLIBRI_E_DEVICE when the kernels set
 * the device error flag (an id out of range or repeated; out is then undefined);
 * COLIBRI_E_INVAL / COLIBRI_E_NOMEM for bad arguments or a short workspace (nothing is
 * enqueued); COLIBRI_E_CUDA when a copy or launch fails. On every return the stream has
 * finished reading the host buffers. T == 0 is a no-op.
 * colibri_moe_host_workspace_bytes: the device workspace the call needs for up to T_max
 * tokens (0 on a bad configuration). */
size_t colibri_moe_host_workspace_bytes(const colibri_layer_cfg *cfg, int T_max);
int colibri_moe_layer_host(const colibri_layer_cfg *cfg, const float *x, int T, const float *Wr,
                           const float *bias, const colibri_expert *experts,
                           const colibri_expert *shared, int32_t *ids, float *w, int ids_given,
                           float *out, void *workspace, size_t ws_bytes, void *stream);

/* Reads the device error flag of a workspace after synchronising `stream`, and clears
 * it. *status_out = COLIBRI_OK or COLIBRI_E_DEVICE. */
int colibri_workspace_status(const colibri_layer_cfg *cfg, int T_max, void *workspace,
                             int *status_out, void *stream);

/* Byte offsets of the layer's intermediates inside its workspace, for inspection by
 * tests (q8 codes of x, bucket lists, h codes, per-pair expert outputs). Valid after a
 * colibri_moe_layer call with the same cfg and T_max. */
typedef struct {
    size_t qx;      /* int8 [T][d]          q8 codes of x */
    size_t sx;      /* fp32 [T][d/32]       their scales */
    size_t offsets; /* int32 [E+1]          bucket offsets (exclusive scan of counts) */
    size_t pairs;   /* int32 [T*k]          pairs p = t*k+i sorted by (expert, p) */
    size_t hq;      /* int8 [T*k+T][fmax]   q8 codes of h per pair (routed, then shared;
                       decode, T <= 32) */
    size_t hs;      /* fp32 [T*k+T][hs_stride] their scales */
    size_t y;       /* fp32 [T*k+T][d]      per-pair expert outputs */
    size_t fmax;    /* row stride of hq: max(ffn, shared_ffn) */
    size_t hs_stride; /* floats per row of hs: fmax/32, rounded up to 4 for decode */
    size_t hbf;     /* prefill (T > 32): uint16 [T*k+T][fmax], the q8 codes of h as bf16;
                       inside each run of 8, element k of the run sits at 2*(k%4) + k/4 */
} colibri_workspace_view;
int colibri_moe_workspace_view(const colibri_layer_cfg *cfg, int T_max, colibri_workspace_view *out);

/* Profiling hook (process-wide, not thread-safe, off by default). While enabled,
 * colibri_moe_layer and colibri_moe_layer_f32 record timing events on their stream around
 * their kernels (seven slots;
 * also under CUDA-graph capture, as external event-record nodes), on the device that
 * was current when profiling was enabled. */
#define COLIBRI_PROFILE_KERNELS 7
int colibri_moe_profile_enable(int on);

/* Milliseconds of each step of the most recent profiled call, after waiting for it:
 * ms[0] q8 of x, [1] router logits, [2] router selection, [3] bucketing, [4] gate/up,
 * [5] down, [6] combine. Steps fused into one kernel report their time in the first of
 * their slots; skipped and fused-away slots read about 0 (the time of an event record).
 * Decode (T <= 32): [1] the routing kernel (router logits and scores with q8, or q8 alone
 * when ids_given), [4] the expert kernel (selection, bucketing, gate/up, down, combine).
 * Prefill: [1] q8 and the router logits, [2] selection, [3] bucketing, [4] and [5] the two
 * GEMMs, [6] combine. colibri_moe_layer_f32: [1] router logits, [2] selection, [4] gate/up,
 * [5] down, [6] combine. The events serialise the kernels (no programmatic overlap).
 * n must be >= COLIBRI_PROFILE_KERNELS. */
int colibri_moe_profile_read(float *ms, int n);

/* Test export: int32 group dots of a packed int4 matrix with one int8 vector, computed
 * by the decode GEMVs' integer dot code.
 *   w device, [rows][cols] in the stored layout (rows % 32 == 0), qa device int8 [cols],
 *   dots device int32 [rows][cols/32] (row-major). */
int colibri_debug_group_dots(const uint8_t *w, const int8_t *qa, int rows, int cols,
                             int32_t *dots, void *stream);

/* Test export: D = A B^T for one tile of integer codes on the tcgen05 tensor core, as the
 * prefill grouped GEMM computes its per-group dots: the codes enter a kind::f16 MMA as
 * bf16 (every integer in [-128, 127] is exact in bf16) and accumulate in fp32 in tensor
 * memory, which is exact for these ranges. (The integer MMA, tcgen05.mma kind::i8, does
 * not exist on sm_103a: ptxas answers "Feature '.kind::i8' not supported on .target
 * 'sm_103a'".)
 *   a device int8 [128][k] (values in [-128, 127]), b device int8 [n][k], row-major;
 *   d device int32 [128][n] (out). n % 16 == 0, n <= 256; k % 16 == 0, k <= 256. */
int colibri_debug_umma_codes(const int8_t *a, const int8_t *b, int n, int k, int32_t *d, void *stream);

/* ---- HBM expert cache -------------------------------------------------------------
 * Experts stream from a larger, slower tier into a small LRU cache of HBM slots
 * (dashen-tech guide, bullet "Streaming d'experts" and section "Router-Lookahead
 * prefetch"; kongchang.com article, section 三级存储分层). Here the slower tier is
 * pinned host memory holding n_layers * n_exp blobs; a miss or a prefetch copies a blob
 * into a slot with cudaMemcpyAsync on the cache's copy stream, and the compute stream
 * waits on the slot's ready event. */
typedef struct colibri_cache colibri_cache;

typedef struct {
    int64_t lookups;         /* ids looked up */
    int64_t hits;            /* ... found resident or already in flight */
    int64_t misses;          /* ... staged on demand */
    int64_t prefetch_staged; /* blobs staged by colibri_expert_cache_stage */
    int64_t prefetch_used;   /* prefetched blobs later hit by a lookup */
    int64_t prefetch_skipped;/* prefetches dropped: every slot pinned */
    int64_t evictions;
    int64_t bytes_staged;    /* host -> HBM bytes enqueued */
    int64_t prefetch_throttled; /* prefetches dropped: the cap on prefetch copies in flight */
    int64_t prefetch_cancelled; /* queued prefetches dropped unfinished (wrong guess or evicted) */
    int64_t prefetch_bytes;  /* host -> HBM bytes enqueued by prefetches (chunks included) */
    int n_slots;
} colibri_cache_stats;

/* Creates a cache.
 *   hbm_pool     device memory owned by the caller, 256-byte aligned; the cache keeps
 *                its per-layer expert tables at its start and cuts the rest into
 *                slots of colibri_blob_layout_for(d, ffn).nbytes
 *   pinned_host  page-locked host memory holding blob (l, e) at offset
 *                (l * n_exp + e) * nbytes
 *   copy_stream  stream for the staging copies (cudaStream_t as void*)
 * Returns COLIBRI_E_NOMEM when the pool holds fewer slots than top_k. */
int colibri_expert_cache_init(colibri_cache **out, void *hbm_pool, size_t pool_bytes,
                              const void *pinned_host, int n_layers, int n_exp, int d, int ffn,
                              int top_k, void *copy_stream);

/* Prefetch: stage the blobs of layer `layer` named by host ids [n] that are not
 * resident (the router-lookahead prefetch of the dashen-tech guide). Resident ones
 * become most recently used. Returns at once. By default the copies are enqueued now on
 * the copy stream; colibri_expert_cache_set_prefetch moves them to a prefetch stream, or
 * queues them as chunks that colibri_expert_cache_wait enqueues. */
int colibri_expert_cache_stage(colibri_cache *c, int layer, const int32_t *ids, int n);

/* Makes the blobs of layer `layer` named by host ids [n] usable by work enqueued on
 * `wait_on` after this call: misses are staged now on the copy stream (or
 * COLIBRI_E_MISS in strict mode), and `wait_on` waits for each slot's ready event.
 * Queued prefetches of `layer` are settled first: a named id's blob is finished on the
 * copy stream (its remaining chunks), the others are cancelled and their slots freed. The slots stay pinned until the
 * next lookup, which also records when the previous batch's compute has finished
 * using them. Afterwards colibri_expert_cache_table(c, layer)[id] holds the expert. */
int colibri_expert_cache_lookup(colibri_cache *c, int layer, const int32_t *ids, int n,
                                void *wait_on);

/* Device table of n_exp colibri_expert for `layer` (entries valid for looked-up ids). */
const colibri_expert *colibri_expert_cache_table(colibri_cache *c, int layer);

/* Usage-pinned hot set (the "self-learning" cache of the kongchang.com article, section
 * 三级存储分层, where learned-hot experts stay in the fast tier): every lookup counts a
 * use of its (layer, id); up to n_hot slots hold the keys with the most uses and are never
 * evicted. A key enters the hot set when there is room or when it has strictly more uses
 * than the weakest hot key (fewest uses, then least recently used), which leaves the set
 * but stays resident. Prefetches do not count as uses. 0 (the default) is plain LRU.
 * COLIBRI_E_INVAL unless 0 <= n_hot <= slots - top_k (a lookup batch must always fit). */
int colibri_expert_cache_set_hot(colibri_cache *c, int n_hot);

/* How prefetches (colibri_expert_cache_stage) are copied. They go on `prefetch_stream`
 * (a cudaStream_t owned by the caller; NULL: the copy stream, as by default), so that a
 * demand miss of colibri_expert_cache_lookup, on the copy stream, never waits behind a
 * speculative copy.
 *   chunk_bytes 0: each prefetch is one whole-blob copy enqueued by stage();
 *     max_in_flight > 0 caps the prefetch copies still running: a prefetch of a
 *     non-resident id beyond the cap is dropped (counted in prefetch_throttled);
 *     0: no cap.
 *   chunk_bytes > 0: stage() only reserves a slot and queues the blob;
 *     colibri_expert_cache_wait enqueues it in chunks of chunk_bytes, at most
 *     max_in_flight (1..64) chunks running, and only while no demand copy runs; a lookup
 *     of the blob's layer finishes it or cancels it. A wrong guess then costs the chunks
 *     already copied, which ran while the copy link was otherwise idle.
 * COLIBRI_E_INVAL for a bad argument, or while queued prefetches or chunks are pending. */
int colibri_expert_cache_set_prefetch(colibri_cache *c, void *prefetch_stream, int max_in_flight,
                                      size_t chunk_bytes);

/* Waits, polling on the calling thread, at most timeout_ms, for the work enqueued so far
 * on `stream` (a cudaStream_t; typically the compute stream, whose current layer decides
 * the next lookup's ids). Meanwhile it enqueues queued prefetch chunks whenever no demand
 * copy is running (the pages' lookahead thread, run while the host waits anyway).
 * COLIBRI_E_TIMEOUT if the work is still running. */
int colibri_expert_cache_wait(colibri_cache *c, void *stream, int timeout_ms);

/* One step of that wait's work, for callers with a wait loop of their own: enqueues up to
 * max_chunks queued prefetch chunks now, if no demand copy is running and fewer than the
 * cap are in flight; *enqueued counts them (0 with chunk_bytes 0 or an empty queue). */
int colibri_expert_cache_pump(colibri_cache *c, int max_chunks, int *enqueued);

/* 1: lookups of non-resident ids fail with COLIBRI_E_MISS instead of staging. */
int colibri_expert_cache_set_strict(colibri_cache *c, int strict);

int colibri_expert_cache_stats(colibri_cache *c, colibri_cache_stats *out);

/* Waits (polling, at most timeout_ms) for every staging copy issued so far, on the copy
 * stream and on the prefetch stream.
 * COLIBRI_E_TIMEOUT if they are still running. */
int colibri_expert_cache_sync(colibri_cache *c, int timeout_ms);

void colibri_expert_cache_destroy(colibri_cache *c);

/* Test hook: the next `count` staging copies fail on the host (no copy is issued) and
 * report COLIBRI_E_STAGE. */
int colibri_expert_cache_inject_stage_failure(colibri_cache *c, int count);

/* Host-only test export of the cache's replacement policy, on abstract keys. ops:
 * kind 0 = start of a lookup batch (unpins every key), 1 = lookup key (pins it),
 * 2 = prefetch key. result: kind 1: 1 hit, 0 miss (inserted), 2 no unpinned slot;
 * kind 2: 1 resident, 0 inserted, 2 no room (skipped); kind 0: 0. */
int colibri_lru_trace(int capacity, int64_t n_ops, const int32_t *kind, const int64_t *key,
                      int8_t *result);

/* colibri_lru_trace with n_hot usage-pinned slots (colibri_expert_cache_set_hot); lookups
 * (kind 1) count as uses, prefetches (kind 2) do not. 0 <= n_hot <= capacity. */
int colibri_lru_trace_hot(int capacity, int n_hot, int64_t n_ops, const int32_t *kind, const int64_t *key,
                          int8_t *result);

#ifdef __cplusplus
}
#endif
#endif
