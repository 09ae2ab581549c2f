// C ABI entry points of libcolibri.so (declared in include/colibri.h).
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "kernels.cuh"
#include "workspace.h"

using namespace clb;

namespace {

inline bool aligned(const void *p, size_t a)
{
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

inline int cuda_status(cudaError_t e)
{
    return e == cudaSuccess ? COLIBRI_OK : COLIBRI_E_CUDA;
}

// Profiling hook state: one event before the first kernel and one after each kernel.
struct Profile {
    bool on = false;
    int device = -1;
    cudaEvent_t ev[COLIBRI_PROFILE_KERNELS + 1] = {};
};
Profile g_prof;

inline int prof_mark(int i, cudaStream_t s)
{
    if (!g_prof.on)
        return COLIBRI_OK;
    return cuda_status(cudaEventRecordWithFlags(g_prof.ev[i], s, cudaEventRecordExternal));
}

}  // namespace

namespace clb {

bool cfg_valid(const colibri_layer_cfg *c)
{
    if (!c || (c->group != 32 && c->group != 64))
        return false;
    const int gq = c->group;
    if (c->d <= 0 || c->d % gq || c->d > 8192 || c->ffn <= 0 || c->ffn % gq || c->ffn > 4096)
        return false;
    if (c->n_exp <= 0 || c->n_exp > 1024 || c->top_k <= 0 || c->top_k > 32 || c->top_k > c->n_exp)
        return false;
    if (c->has_shared && (c->shared_ffn <= 0 || c->shared_ffn % gq || c->shared_ffn > 4096))
        return false;
    if (c->router == COLIBRI_ROUTER_SIGMOID_GROUPED) {
        if (c->n_group <= 0 || c->n_group > 32 || c->n_exp % c->n_group)
            return false;
        if (c->topk_group <= 0 || c->topk_group > c->n_group)
            return false;
        if (c->topk_group * (c->n_exp / c->n_group) < c->top_k)
            return false;
    } else if (c->router != COLIBRI_ROUTER_SOFTMAX) {
        return false;
    }
    return true;
}

// Batches above DECODE_T_MAX tokens take the tensor-core grouped GEMMs, whose row tiles
// are 128 rows; other shapes stay on the decode kernels (which chunk any token count).
bool uses_gemm(const colibri_layer_cfg *c, int T)
{
    return T > DECODE_T_MAX && c->d % 128 == 0 && c->ffn % 128 == 0 &&
           (!c->has_shared || c->shared_ffn % 128 == 0);
}

static size_t up256(size_t n)
{
    return (n + 255) & ~size_t(255);
}

WsLayout ws_layout(const colibri_layer_cfg *c, int T, bool stack)
{
    WsLayout L{};
    const size_t d = c->d, E = c->n_exp, K = c->top_k;
    const size_t fmax = c->has_shared && c->shared_ffn > c->ffn ? c->shared_ffn : c->ffn;
    const size_t PT = (size_t)T * K + (c->has_shared ? (size_t)T : 0);
    const size_t nslots = ((size_t)T * K < E ? (size_t)T * K : E) + 1;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = up256(o + bytes);
        return at;
    };
    L.err = take(256);
    L.counters = take(sizeof(Counters));
    L.nslots = nslots;
    // 64-element groups: one pair counter per (row of h, 64-group) for the decode kernel's
    // q8 of h across two gate/up items
    L.hpair_count = c->group == 64 ? PT * (fmax / 64) : 0;
    L.sync_bytes = 4 * (4 + nslots + d / G + L.hpair_count);
    L.sync_stride = (L.sync_bytes + 15) & ~size_t(15);
    L.sync = take(stack ? 2 * L.sync_stride + 16 : L.sync_bytes);
    L.bar = stack ? L.sync + 2 * L.sync_stride : 0;
    L.sync_end = stack ? L.bar + 16 : L.sync + L.sync_bytes;
    L.qx = take((size_t)T * d);
    L.qx_eo = take((size_t)T * d);
    L.sx = take(4 * (size_t)T * (d / G));
    L.xc = take(4 * (size_t)T * (d / G));
    L.logits = take(4 * (size_t)T * E);
    L.s = take(4 * (size_t)T * E);
    L.c = take(4 * (size_t)T * E);
    L.offsets = take(4 * (E + 1));
    L.pairs = take(4 * (size_t)T * K);
    L.slots = take(sizeof(Slot) * nslots);
    L.hq = take(PT * fmax);
    L.hq_eo = take(PT * fmax);
    const size_t hgs = (size_t)decode_hgs((int)fmax);  // >= fmax / G
    L.hs = take(4 * PT * hgs);
    L.hc = take(4 * PT * hgs);
    L.y = take(4 * PT * d);
    const bool prefill = uses_gemm(c, T);
    L.hf = take(c->group == 64 && !prefill ? 4 * PT * fmax : 0);  // fp32 h before its q8 per 64
    L.xbf = take(prefill ? 2 * (size_t)T * d : 0);
    L.hbf = take(prefill ? 2 * PT * fmax : 0);
    L.fmax = fmax;
    L.total = o;
    return L;
}

}  // namespace clb

namespace clb {

// The decode kernel's arguments for one layer; `sync` is its control-word area.
DecodeArgs decode_args(const colibri_layer_cfg *cfg, int T, const WsLayout &L, char *ws, const float *x,
                       const float *Wr, const float *bias, const colibri_expert *experts, const colibri_expert &sh,
                       int32_t *ids, float *w, int ids_given, float *out, int *sync)
{
    const int d = cfg->d;
    int *err = reinterpret_cast<int *>(ws + L.err);
    float *lg = reinterpret_cast<float *>(ws + L.logits);
    float *sv = reinterpret_cast<float *>(ws + L.s);
    float *cv = reinterpret_cast<float *>(ws + L.c);
    DecodeArgs da{};
    da.experts = experts;
    da.shared = sh;
    da.d = d;
    da.ffn = cfg->ffn;
    da.shared_ffn = cfg->shared_ffn;
    da.T = T;
    da.K = cfg->top_k;
    da.has_shared = cfg->has_shared;
    da.fmax = (int)L.fmax;
    da.x = x;
    da.Wr = ids_given ? nullptr : Wr;
    da.bias = cfg->router == COLIBRI_ROUTER_SOFTMAX ? nullptr : bias;
    da.ids_given = ids_given ? 1 : 0;
    da.E = cfg->n_exp;
    da.n_group = cfg->router == COLIBRI_ROUTER_SOFTMAX ? 1 : cfg->n_group;
    da.topk_group = cfg->router == COLIBRI_ROUTER_SOFTMAX ? 1 : cfg->topk_group;
    da.router = cfg->router;
    da.norm_topk = cfg->norm_topk;
    da.routed_scale = cfg->routed_scale;
    da.logits = lg;
    da.rs = sv;
    da.rc = cv;
    da.ids = ids;
    da.w_in = w;
    da.w_out = w;
    da.offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    da.pairs = reinterpret_cast<int32_t *>(ws + L.pairs);
    da.slots = reinterpret_cast<Slot *>(ws + L.slots);
    da.counters = reinterpret_cast<Counters *>(ws + L.counters);
    da.qx = reinterpret_cast<int8_t *>(ws + L.qx);
    da.xq_eo = reinterpret_cast<int8_t *>(ws + L.qx_eo);
    da.sx = reinterpret_cast<float *>(ws + L.sx);
    da.xc = reinterpret_cast<int *>(ws + L.xc);
    da.hq = reinterpret_cast<int8_t *>(ws + L.hq);
    da.hq_eo = reinterpret_cast<int8_t *>(ws + L.hq_eo);
    da.hs = reinterpret_cast<float *>(ws + L.hs);
    da.hc = reinterpret_cast<int *>(ws + L.hc);
    da.y = reinterpret_cast<float *>(ws + L.y);
    da.out = out;
    da.claim = sync;
    da.route_done = sync + 1;
    da.done_gu = sync + 4;
    da.done_rb = sync + 4 + L.nslots;
    da.err = err;
    da.max_slots = (int)L.nslots;
    da.group = cfg->group;
    da.hf = reinterpret_cast<float *>(ws + L.hf);
    da.hpair = sync + 4 + L.nslots + d / G;
    return da;
}

}  // namespace clb

extern "C" {

int colibri_blob_layout_for(int d, int f, colibri_blob_layout *out)
{
    return colibri_blob_layout_for_g(d, f, COLIBRI_GROUP, out);
}

int colibri_blob_layout_for_g(int d, int f, int group, colibri_blob_layout *out)
{
    if (!out || (group != 32 && group != 64) || d <= 0 || f <= 0 || d % group || f % group)
        return COLIBRI_E_INVAL;
    const size_t nib = (size_t)f * d / 2, sc = 4 * (size_t)f * (d / group);
    const size_t nib2 = (size_t)d * f / 2, sc2 = 4 * (size_t)d * (f / group);
    size_t o = 0;
    out->w1 = o;
    o = up256(o + nib);
    out->w3 = o;
    o = up256(o + nib);
    out->w2 = o;
    o = up256(o + nib2);
    out->s1 = o;
    o = up256(o + sc);
    out->s3 = o;
    o = up256(o + sc);
    out->s2 = o;
    o = up256(o + sc2);
    out->nbytes = o;
    return COLIBRI_OK;
}

const char *colibri_strerror(int status)
{
    switch (status) {
    case COLIBRI_OK: return "ok";
    case COLIBRI_E_INVAL: return "invalid argument or configuration";
    case COLIBRI_E_CUDA: return "CUDA runtime error";
    case COLIBRI_E_NOMEM: return "workspace or cache pool too small";
    case COLIBRI_E_TIMEOUT: return "bounded wait ran out";
    case COLIBRI_E_MISS: return "expert not resident (strict cache)";
    case COLIBRI_E_STAGE: return "staging an expert failed";
    case COLIBRI_E_DEVICE: return "a kernel reported bad input";
    default: return "unknown status";
    }
}

int colibri_q8_quantize(const float *x, int rows, int cols, int8_t *q, float *scale, void *stream)
{
    return colibri_q8_quantize_g(x, rows, cols, COLIBRI_GROUP, q, scale, stream);
}

int colibri_q8_quantize_g(const float *x, int rows, int cols, int group, int8_t *q, float *scale, void *stream)
{
    if (rows < 0 || cols <= 0 || (group != 32 && group != 64) || cols % group)
        return COLIBRI_E_INVAL;
    if (rows == 0)
        return COLIBRI_OK;
    if (!x || !q || !scale)
        return COLIBRI_E_INVAL;
    Q8Args a{x, rows, cols, q, scale, nullptr, nullptr, nullptr, group};  // codes and scales only
    const long groups = (long)rows * (cols / group);
    const long blocks = (groups + 7) / 8;
    if (blocks > 0x7fffffffL)
        return COLIBRI_E_INVAL;
    k_q8<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(a);
    return cuda_status(cudaGetLastError());
}

// Raises a kernel's dynamic shared memory limit to `bytes` whenever a launch needs more
// than the largest limit set so far (the limits only grow). The default limit covers
// 48 KB of static plus dynamic shared memory together, so even a launch just under it
// sets the attribute.
// Tracked per device: the attribute belongs to the device's context. Host threads that
// launch at the same time take the lock, so the attribute and the record of it agree.
constexpr int kMaxDev = 64;
struct SmemLimits {
    std::mutex mu;
    size_t have[kMaxDev] = {};
};

static bool smem_attr(const void *fn, size_t bytes, SmemLimits &lim)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
        return false;
    std::lock_guard<std::mutex> lock(lim.mu);
    if (bytes <= lim.have[dev])
        return true;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
        return false;
    lim.have[dev] = bytes;
    return true;
}

// Token rows of x that k_route_logits stages per pass: up to 96 KB of x, at least one row.
static int route_xt(int d, int T)
{
    int xt = (96 * 1024) / (d * 4);
    xt = xt < 1 ? 1 : xt;
    xt = xt > 32 ? 32 : xt;
    return xt > T ? T : xt;
}

// Router logits (+ s and c when s_arr is given, + q8 of x when q8.x is set).
static int launch_route_logits(const colibri_layer_cfg *cfg, const float *x, int T, const float *Wr,
                               const float *bias, float *logits, float *s_arr, float *c_arr,
                               const Q8Args &q8, int *err, cudaStream_t s)
{
    static SmemLimits have;
    const int xt = route_xt(cfg->d, T);
    const size_t smem = (size_t)cfg->d * 4 * (size_t)(1 + xt);
    const bool sig = cfg->router != COLIBRI_ROUTER_SOFTMAX;
    RouterArgs ra{x, T, cfg->d, cfg->n_exp, xt, Wr, sig ? bias : nullptr, logits,
                  sig ? s_arr : nullptr, sig ? c_arr : nullptr, q8, err};
    if (T > DECODE_T_MAX) {
        // many tokens: (token x expert) tiles; q8 of x runs as its own kernel
        if (q8.x) {
            const long groups = (long)T * (cfg->d / cfg->group);
            k_q8<<<(unsigned)((groups + 7) / 8), 256, 0, s>>>(q8);
            if (cudaGetLastError() != cudaSuccess)
                return COLIBRI_E_CUDA;
        }
        ra.q8.x = nullptr;
        static SmemLimits have_tiled;
        if (!smem_attr((const void *)k_route_logits_tiled, ROUTE_TILED_SMEM, have_tiled))
            return COLIBRI_E_CUDA;
        dim3 grid((T + 15) / 16, (cfg->n_exp + 31) / 32);
        k_route_logits_tiled<<<grid, 256, ROUTE_TILED_SMEM, s>>>(ra);
        return cuda_status(cudaGetLastError());
    }
    if (!smem_attr((const void *)k_route_logits, smem, have))
        return COLIBRI_E_CUDA;
    k_route_logits<<<cfg->n_exp, 128, smem, s>>>(ra);
    return cuda_status(cudaGetLastError());
}

static SelectArgs select_args(const colibri_layer_cfg *cfg, int T, const float *logits, const float *s_arr,
                              const float *c_arr, const float *bias, int32_t *ids, float *w)
{
    const bool sig = cfg->router != COLIBRI_ROUTER_SOFTMAX;
    return SelectArgs{logits, sig ? s_arr : nullptr, sig ? c_arr : nullptr, sig ? bias : nullptr, T,
                      cfg->n_exp, cfg->top_k, cfg->n_group, cfg->topk_group, cfg->router, cfg->norm_topk,
                      cfg->routed_scale, ids, w};
}

static int launch_select(const SelectArgs &sa, cudaStream_t s)
{
    constexpr int SEL_WARPS = 4;
    k_router_select<<<(sa.T + SEL_WARPS - 1) / SEL_WARPS, 32 * SEL_WARPS, 0, s>>>(sa);
    return cuda_status(cudaGetLastError());
}

static int launch_router(const colibri_layer_cfg *cfg, const float *x, int T, const float *Wr,
                         const float *bias, float *logits, int32_t *ids, float *w, cudaStream_t s)
{
    const Q8Args none{};
    int rc = launch_route_logits(cfg, x, T, Wr, bias, logits, nullptr, nullptr, none, nullptr, s);
    if (rc)
        return rc;
    return launch_select(select_args(cfg, T, logits, nullptr, nullptr, bias, ids, w), s);
}

int colibri_router_topk(const colibri_layer_cfg *cfg, const float *x, int T, const float *Wr,
                        const float *bias, float *logits, int32_t *ids, float *w, void *stream)
{
    if (!cfg_valid(cfg) || T < 0)
        return COLIBRI_E_INVAL;
    if (T == 0)
        return COLIBRI_OK;
    if (!x || !Wr || !logits || !ids || !w || !aligned(Wr, 16) || !aligned(x, 16))
        return COLIBRI_E_INVAL;
    return launch_router(cfg, x, T, Wr, bias, logits, ids, w, (cudaStream_t)stream);
}

size_t colibri_moe_workspace_bytes(const colibri_layer_cfg *cfg, int T_max)
{
    if (!cfg_valid(cfg) || T_max < 0)
        return 0;
    return ws_layout(cfg, T_max).total;
}

int colibri_moe_workspace_view(const colibri_layer_cfg *cfg, int T_max, colibri_workspace_view *out)
{
    if (!cfg_valid(cfg) || T_max < 0 || !out)
        return COLIBRI_E_INVAL;
    const WsLayout L = ws_layout(cfg, T_max);
    out->qx = L.qx;
    out->sx = L.sx;
    out->offsets = L.offsets;
    out->pairs = L.pairs;
    out->hq = L.hq;
    out->hs = L.hs;
    out->y = L.y;
    out->fmax = L.fmax;
    out->hs_stride = uses_gemm(cfg, T_max) ? L.fmax / cfg->group : (size_t)decode_hgs((int)L.fmax);
    out->hbf = L.hbf;
    return COLIBRI_OK;
}

int colibri_workspace_status(const colibri_layer_cfg *cfg, int T_max, void *workspace,
                             int *status_out, void *stream)
{
    if (!cfg_valid(cfg) || !workspace || !status_out)
        return COLIBRI_E_INVAL;
    const WsLayout L = ws_layout(cfg, T_max);
    int flag = 0;
    cudaStream_t s = (cudaStream_t)stream;
    char *ws = static_cast<char *>(workspace);
    if (cudaMemcpyAsync(&flag, ws + L.err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return COLIBRI_E_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return COLIBRI_E_CUDA;
    if (flag && cudaMemsetAsync(ws + L.err, 0, sizeof(int), s) != cudaSuccess)
        return COLIBRI_E_CUDA;
    *status_out = flag ? COLIBRI_E_DEVICE : COLIBRI_OK;
    return COLIBRI_OK;
}

int colibri_moe_layer(const colibri_layer_cfg *cfg, const float *x, int T, const float *Wr,
                      const float *bias, const colibri_expert *experts,
                      const colibri_expert *shared, int32_t *ids, float *w, int ids_given,
                      float *out, void *workspace, size_t ws_bytes, void *stream)
{
    if (!cfg_valid(cfg) || T < 0)
        return COLIBRI_E_INVAL;
    if (T == 0)
        return COLIBRI_OK;
    if (!x || !experts || !ids || !w || !out || !workspace)
        return COLIBRI_E_INVAL;
    if (cfg->has_shared && !shared)
        return COLIBRI_E_INVAL;
    if (!ids_given && (!Wr || !aligned(Wr, 16)))
        return COLIBRI_E_INVAL;
    if (!aligned(workspace, 256) || !aligned(out, 16) || !aligned(x, 16))
        return COLIBRI_E_INVAL;
    const WsLayout L = ws_layout(cfg, T);
    if (ws_bytes < L.total)
        return COLIBRI_E_NOMEM;
    cudaStream_t s = (cudaStream_t)stream;
    char *ws = static_cast<char *>(workspace);
    int *err = reinterpret_cast<int *>(ws + L.err);
    const int d = cfg->d, E = cfg->n_exp, K = cfg->top_k;

    // the control words (error flag, routing counter), the work counters and the decode
    // kernel's claim and completion counters start every call at zero: if routing fails,
    // the expert kernels find no work
    if (cudaMemsetAsync(ws + L.err, 0, L.sync_end - L.err, s) != cudaSuccess)
        return COLIBRI_E_CUDA;
    if (prof_mark(0, s))
        return COLIBRI_E_CUDA;
    const bool prefill = uses_gemm(cfg, T);
    // q8 of x for prefill: plain codes and scales, and the bf16 codes in the tensor-core
    // order (decode quantises x inside its kernel)
    Q8Args qa{x, T, d, reinterpret_cast<int8_t *>(ws + L.qx), reinterpret_cast<float *>(ws + L.sx), nullptr,
              nullptr, reinterpret_cast<uint16_t *>(ws + L.xbf), cfg->group};
    const int down_blocks = (d + DN_ITEM_ROWS - 1) / DN_ITEM_ROWS;
    BucketArgs ba{ids, T, K, E, cfg->has_shared, cfg->shared_ffn, cfg->ffn, down_blocks, 0,
                  reinterpret_cast<int32_t *>(ws + L.offsets), reinterpret_cast<int32_t *>(ws + L.pairs),
                  reinterpret_cast<Slot *>(ws + L.slots), reinterpret_cast<Counters *>(ws + L.counters), err};
    float *lg = reinterpret_cast<float *>(ws + L.logits);
    float *sv = reinterpret_cast<float *>(ws + L.s);
    float *cv = reinterpret_cast<float *>(ws + L.c);
    const SelectArgs sa = select_args(cfg, T, lg, sv, cv, bias, ids, w);
    colibri_expert sh{};
    if (cfg->has_shared)
        sh = *shared;
    if (!prefill) {
        // decode: one kernel for q8 of x, router logits, selection (unless ids_given),
        // bucketing, gate/up, down and the combine
        if (prof_mark(1, s) || prof_mark(2, s) || prof_mark(3, s) || prof_mark(4, s))
            return COLIBRI_E_CUDA;
        const DecodeArgs da = decode_args(cfg, T, L, ws, x, Wr, bias, experts, sh, ids, w, ids_given, out,
                                          reinterpret_cast<int *>(ws + L.sync));
        if (launch_decode(da, s) != cudaSuccess || prof_mark(5, s) || prof_mark(6, s) || prof_mark(7, s))
            return COLIBRI_E_CUDA;
        return COLIBRI_OK;
    }
    if (ids_given) {
        // a1: q8 of x
        const long groups = (long)T * (d / cfg->group);
        k_q8<<<(unsigned)((groups + 7) / 8), 256, 0, s>>>(qa);
        if (cudaGetLastError() != cudaSuccess || prof_mark(1, s) || prof_mark(2, s) || prof_mark(3, s))
            return COLIBRI_E_CUDA;
    } else {
        // a1-a3: router logits with sigmoid scores, q8 of x, selection
        if (prof_mark(1, s))
            return COLIBRI_E_CUDA;
        int rc = launch_route_logits(cfg, x, T, Wr, bias, lg, sv, cv, qa, err, s);
        if (rc || prof_mark(2, s))
            return COLIBRI_E_CUDA;
        if (launch_select(sa, s) || prof_mark(3, s))
            return COLIBRI_E_CUDA;
    }
    {
        // a4: bucketing and slot list (counters, plus the ids when they fit in 160 KB)
        static SmemLimits have;
        const size_t bsm0 = bucket_smem_bytes(E, 1024), pbytes = (size_t)T * K * sizeof(int);
        ba.stage_ids = bsm0 + pbytes <= 160 * 1024;
        const size_t bsm = bsm0 + (ba.stage_ids ? pbytes : 0);
        if (!smem_attr((const void *)k_bucket, bsm, have))
            return COLIBRI_E_CUDA;
        k_bucket<<<1, 1024, bsm, s>>>(ba);
        if (cudaGetLastError() != cudaSuccess || prof_mark(4, s))
            return COLIBRI_E_CUDA;
    }
    // a10-a11: grouped GEMMs on the tensor cores
    GemmArgs gm{};
    gm.experts = experts;
    gm.shared = sh;
    gm.d = d;
    gm.ffn = cfg->ffn;
    gm.shared_ffn = cfg->shared_ffn;
    gm.T = T;
    gm.K = K;
    gm.has_shared = cfg->has_shared;
    gm.fmax = (int)L.fmax;
    gm.slots = reinterpret_cast<const Slot *>(ws + L.slots);
    gm.counters = reinterpret_cast<const Counters *>(ws + L.counters);
    gm.pairs = reinterpret_cast<const int32_t *>(ws + L.pairs);
    gm.group = cfg->group;
    gm.err = err;
    GemmArgs gg = gm;
    gg.abf = reinterpret_cast<const uint16_t *>(ws + L.xbf);
    gg.as = reinterpret_cast<const float *>(ws + L.sx);
    gg.act_stride = d;
    gg.act_groups = d / cfg->group;
    gg.hbf = reinterpret_cast<uint16_t *>(ws + L.hbf);
    gg.hs = reinterpret_cast<float *>(ws + L.hs);
    if (launch_gemm(MODE_GATEUP, gg, s) != cudaSuccess || prof_mark(5, s))
        return COLIBRI_E_CUDA;
    GemmArgs gd = gm;
    gd.abf = reinterpret_cast<const uint16_t *>(ws + L.hbf);
    gd.as = reinterpret_cast<const float *>(ws + L.hs);
    gd.act_stride = (long)L.fmax;
    gd.act_groups = (int)L.fmax / cfg->group;
    gd.y = reinterpret_cast<float *>(ws + L.y);
    if (launch_gemm(MODE_DOWN, gd, s) != cudaSuccess || prof_mark(6, s))
        return COLIBRI_E_CUDA;

    // a9: combine
    CombineArgs ca{reinterpret_cast<const float *>(ws + L.y), w, T, K, d, cfg->has_shared, out};
    dim3 cg((d / 4 + 255) / 256, T);
    k_combine<<<cg, 256, 0, s>>>(ca);
    if (cudaGetLastError() != cudaSuccess || prof_mark(7, s))
        return COLIBRI_E_CUDA;
    return COLIBRI_OK;
}

size_t colibri_moe_stack_workspace_bytes(const colibri_layer_cfg *cfg, int T_max)
{
    if (!cfg_valid(cfg) || T_max < 0 || T_max > DECODE_T_MAX)
        return 0;
    return ws_layout(cfg, T_max, true).total;
}

int colibri_moe_stack_decode(const colibri_layer_cfg *cfg, const float *x, int T, int n_layers,
                             const colibri_stack_layer *layers, int ids_given, void *workspace,
                             size_t ws_bytes, void *stream)
{
    if (!cfg_valid(cfg) || T < 0 || T > DECODE_T_MAX || n_layers < 1 || n_layers > COLIBRI_STACK_MAX ||
        !layers)
        return COLIBRI_E_INVAL;
    if (T == 0)
        return COLIBRI_OK;
    if (!workspace || !aligned(workspace, 256))
        return COLIBRI_E_INVAL;
    // layer l's activations: its own x, else the previous layer's out (x for layer 0)
    auto input_of = [&](int l) -> const float * {
        return layers[l].x ? layers[l].x : l ? layers[l - 1].out : x;
    };
    for (int l = 0; l < n_layers; ++l) {
        const colibri_stack_layer &y = layers[l];
        if (!input_of(l) || !aligned(input_of(l), 16))
            return COLIBRI_E_INVAL;
        if (!y.experts || !y.ids || !y.w || !y.out || !aligned(y.out, 16))
            return COLIBRI_E_INVAL;
        if (cfg->has_shared && !y.shared)
            return COLIBRI_E_INVAL;
        if (!ids_given && (!y.Wr || !aligned(y.Wr, 16)))
            return COLIBRI_E_INVAL;
        // layer l reads its input while it writes its output
        if (y.out == input_of(l))
            return COLIBRI_E_INVAL;
    }
    const WsLayout L = ws_layout(cfg, T, true);
    if (ws_bytes < L.total)
        return COLIBRI_E_NOMEM;
    cudaStream_t s = (cudaStream_t)stream;
    char *ws = static_cast<char *>(workspace);
    // the error word, both control-word areas and the barrier start at zero
    if (cudaMemsetAsync(ws + L.err, 0, L.sync_end - L.err, s) != cudaSuccess)
        return COLIBRI_E_CUDA;
    DecodeStack p{};
    p.L = n_layers;
    p.bar = reinterpret_cast<int *>(ws + L.bar);
    p.sync_area[0] = reinterpret_cast<int *>(ws + L.sync);
    p.sync_area[1] = reinterpret_cast<int *>(ws + L.sync + L.sync_stride);
    p.sync_words = (int)(L.sync_stride / 4);
    for (int l = 0; l < n_layers; ++l) {
        const colibri_stack_layer &y = layers[l];
        colibri_expert sh{};
        if (cfg->has_shared)
            sh = *y.shared;
        p.layer[l] = decode_args(cfg, T, L, ws, input_of(l), y.Wr, y.bias, y.experts, sh, y.ids, y.w, ids_given,
                                 y.out, p.sync_area[l & 1]);
    }
    return launch_decode_stack(p, s) == cudaSuccess ? COLIBRI_OK : COLIBRI_E_CUDA;
}

// Workspace of colibri_moe_layer_f32: error flag | logits [T][E] | sigmoid scores s and
// biased scores c [T][E] | h [PT][fmax] | y [PT][d], PT = T*K (+ T with a shared expert),
// each part 256-byte aligned. The error flag sits at offset 0, as in colibri_moe_layer's
// workspace.
struct F32Layout {
    size_t err, logits, s, c, h, y, fmax, pt, total;
};

static F32Layout f32_layout(const colibri_layer_cfg *c, int T)
{
    F32Layout L{};
    L.fmax = c->has_shared && c->shared_ffn > c->ffn ? c->shared_ffn : c->ffn;
    L.pt = (size_t)T * c->top_k + (c->has_shared ? (size_t)T : 0);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = (o + bytes + 255) & ~size_t(255);
        return at;
    };
    L.err = take(256);
    L.logits = take(4 * (size_t)T * c->n_exp);
    L.s = take(4 * (size_t)T * c->n_exp);
    L.c = take(4 * (size_t)T * c->n_exp);
    L.h = take(4 * L.pt * L.fmax);
    L.y = take(4 * L.pt * c->d);
    L.total = o;
    return L;
}

size_t colibri_moe_f32_workspace_bytes(const colibri_layer_cfg *cfg, int T_max)
{
    if (!cfg_valid(cfg) || T_max < 0 || T_max > DECODE_T_MAX)
        return 0;
    return f32_layout(cfg, T_max).total;
}

int colibri_moe_layer_f32(const colibri_layer_cfg *cfg, const float *x, int T, const float *Wr,
                          const float *bias, const colibri_expert *experts,
                          const colibri_expert *shared, int32_t *ids, float *w, int ids_given,
                          float *out, void *workspace, size_t ws_bytes, void *stream)
{
    if (!cfg_valid(cfg) || T < 0 || T > DECODE_T_MAX)
        return COLIBRI_E_INVAL;
    if (T == 0)
        return COLIBRI_OK;
    if (!x || !experts || !ids || !w || !out || !workspace)
        return COLIBRI_E_INVAL;
    if (cfg->has_shared && !shared)
        return COLIBRI_E_INVAL;
    if (!ids_given && (!Wr || !aligned(Wr, 16)))
        return COLIBRI_E_INVAL;
    if (!aligned(workspace, 256) || !aligned(out, 16) || !aligned(x, 16))
        return COLIBRI_E_INVAL;
    const F32Layout L = f32_layout(cfg, T);
    if (ws_bytes < L.total)
        return COLIBRI_E_NOMEM;
    cudaStream_t s = (cudaStream_t)stream;
    char *ws = static_cast<char *>(workspace);
    int *err = reinterpret_cast<int *>(ws + L.err);
    float *lg = reinterpret_cast<float *>(ws + L.logits);
    if (cudaMemsetAsync(ws + L.err, 0, 256, s) != cudaSuccess)
        return COLIBRI_E_CUDA;
    // profiling slots: as colibri_moe_layer's prefill path (no q8, no bucketing)
    if (prof_mark(0, s) || prof_mark(1, s))
        return COLIBRI_E_CUDA;
    if (!ids_given) {
        // the logits kernel evaluates the sigmoid scores (spread over its CTAs) and hands
        // them to the selection, as on the int8 path
        const Q8Args none{};
        float *sv = reinterpret_cast<float *>(ws + L.s), *cv = reinterpret_cast<float *>(ws + L.c);
        if (launch_route_logits(cfg, x, T, Wr, bias, lg, sv, cv, none, err, s) || prof_mark(2, s))
            return COLIBRI_E_CUDA;
        if (launch_select(select_args(cfg, T, lg, sv, cv, bias, ids, w), s) || prof_mark(3, s))
            return COLIBRI_E_CUDA;
    } else if (prof_mark(2, s) || prof_mark(3, s)) {
        return COLIBRI_E_CUDA;
    }
    if (prof_mark(4, s))
        return COLIBRI_E_CUDA;
    F32Args fa{};
    fa.experts = experts;
    if (cfg->has_shared)
        fa.shared = *shared;
    fa.ids = ids;
    fa.x = x;
    fa.h = reinterpret_cast<float *>(ws + L.h);
    fa.y = reinterpret_cast<float *>(ws + L.y);
    fa.T = T;
    fa.K = cfg->top_k;
    fa.E = cfg->n_exp;
    fa.d = cfg->d;
    fa.ffn = cfg->ffn;
    fa.shared_ffn = cfg->shared_ffn;
    fa.has_shared = cfg->has_shared;
    fa.fmax = (int)L.fmax;
    fa.gsh = cfg->group == 64 ? 1 : 0;
    fa.err = err;
    const unsigned pt = (unsigned)L.pt;
    k_f32_gateup<<<dim3((unsigned)(L.fmax / G), pt), 256, f32_smem_gateup(cfg->d), s>>>(fa);
    if (cudaGetLastError() != cudaSuccess || prof_mark(5, s))
        return COLIBRI_E_CUDA;
    k_f32_down<<<dim3((unsigned)(cfg->d / G), pt), 256, f32_smem_down((int)L.fmax), s>>>(fa);
    if (cudaGetLastError() != cudaSuccess || prof_mark(6, s))
        return COLIBRI_E_CUDA;
    CombineArgs ca{fa.y, w, T, cfg->top_k, cfg->d, cfg->has_shared, out};
    k_combine<<<dim3((unsigned)((cfg->d / 4 + 255) / 256), (unsigned)T), 256, 0, s>>>(ca);
    if (cudaGetLastError() != cudaSuccess || prof_mark(7, s))
        return COLIBRI_E_CUDA;
    return COLIBRI_OK;
}

int colibri_moe_profile_enable(int on)
{
    if (on && !g_prof.ev[0]) {
        if (cudaGetDevice(&g_prof.device) != cudaSuccess)
            return COLIBRI_E_CUDA;
        for (auto &e : g_prof.ev)
            if (cudaEventCreate(&e) != cudaSuccess)
                return COLIBRI_E_CUDA;
    }
    g_prof.on = on != 0;
    return COLIBRI_OK;
}

int colibri_moe_profile_read(float *ms, int n)
{
    if (!ms || n < COLIBRI_PROFILE_KERNELS || !g_prof.ev[0])
        return COLIBRI_E_INVAL;
    if (cudaEventSynchronize(g_prof.ev[COLIBRI_PROFILE_KERNELS]) != cudaSuccess)
        return COLIBRI_E_CUDA;
    for (int i = 0; i < COLIBRI_PROFILE_KERNELS; ++i)
        if (cudaEventElapsedTime(&ms[i], g_prof.ev[i], g_prof.ev[i + 1]) != cudaSuccess)
            return COLIBRI_E_CUDA;
    return COLIBRI_OK;
}

int colibri_debug_umma_codes(const int8_t *a, const int8_t *b, int n, int k, int32_t *d, void *stream)
{
    if (!a || !b || !d || n <= 0 || n % 16 || n > 256 || k <= 0 || k % 16 || k > 256)
        return COLIBRI_E_INVAL;
    static SmemLimits have;
    const size_t smem = debug_umma_smem(n, k);
    if (!smem_attr((const void *)k_debug_umma, smem, have))
        return COLIBRI_E_CUDA;
    k_debug_umma<<<1, 128, smem, (cudaStream_t)stream>>>(a, b, n, k, d, nullptr);
    return cuda_status(cudaGetLastError());
}

int colibri_debug_group_dots(const uint8_t *w, const int8_t *qa, int rows, int cols, int32_t *dots,
                             void *stream)
{
    if (!w || !qa || !dots || rows < 0 || rows % 32 || cols <= 0 || cols % G)
        return COLIBRI_E_INVAL;
    if (rows == 0)
        return COLIBRI_OK;
    if (!aligned(w, 16) || !aligned(qa, 16))
        return COLIBRI_E_INVAL;
    const long n = (long)rows * (cols / G);
    k_debug_dots<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream>>>(w, qa, rows, cols, dots);
    return cuda_status(cudaGetLastError());
}

}  // extern "C"
