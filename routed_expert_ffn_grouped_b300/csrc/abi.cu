// C ABI entry points of libcolibri.so (declared in include/colibri.h).
#include <stdio.h>
#include <string.h>

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
    if (!c || c->group != G)
        return false;
    if (c->d <= 0 || c->d % G || c->d > 8192 || c->ffn <= 0 || c->ffn % G || c->ffn > 4096)
        return false;
    if (c->n_exp <= 0 || c->n_exp > 1024 || c->top_k <= 0 || c->top_k > 32 || c->top_k > c->n_exp)
        return false;
    if (c->has_shared && (c->shared_ffn <= 0 || c->shared_ffn % G || c->shared_ffn > 4096))
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

static size_t up256(size_t n)
{
    return (n + 255) & ~size_t(255);
}

WsLayout ws_layout(const colibri_layer_cfg *c, int T)
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
    L.qx = take((size_t)T * d);
    L.qx_eo = take((size_t)T * d);
    L.sx = take(4 * (size_t)T * (d / G));
    L.xc = take(4 * (size_t)T * (d / G));
    L.logits = take(4 * (size_t)T * E);
    L.offsets = take(4 * (E + 1));
    L.pairs = take(4 * (size_t)T * K);
    L.slots = take(sizeof(Slot) * nslots);
    L.hq = take(PT * fmax);
    L.hq_eo = take(PT * fmax);
    L.hs = take(4 * PT * (fmax / G));
    L.hc = take(4 * PT * (fmax / G));
    L.y = take(4 * PT * d);
    L.fmax = fmax;
    L.total = o;
    return L;
}

}  // namespace clb

extern "C" {

int colibri_blob_layout_for(int d, int f, colibri_blob_layout *out)
{
    if (!out || d <= 0 || f <= 0 || d % G || f % G)
        return COLIBRI_E_INVAL;
    const size_t nib = (size_t)f * d / 2, sc = 4 * (size_t)f * (d / G);
    const size_t nib2 = (size_t)d * f / 2, sc2 = 4 * (size_t)d * (f / G);
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
    if (rows < 0 || cols <= 0 || cols % G)
        return COLIBRI_E_INVAL;
    if (rows == 0)
        return COLIBRI_OK;
    if (!x || !q || !scale)
        return COLIBRI_E_INVAL;
    Q8Args a{x, rows, cols, q, scale, nullptr, nullptr, nullptr};
    const long groups = (long)rows * (cols / G);
    const long blocks = (groups + 7) / 8;
    if (blocks > 0x7fffffffL)
        return COLIBRI_E_INVAL;
    k_q8<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(a);
    return cuda_status(cudaGetLastError());
}

static int launch_router(const colibri_layer_cfg *cfg, const float *x, int T, const float *Wr,
                         const float *bias, float *logits, int32_t *ids, float *w, int *err,
                         cudaStream_t s, int prof_at)
{
    RouterArgs ra{x, T, cfg->d, cfg->n_exp, Wr, logits, err};
    k_router_logits<<<cfg->n_exp, 32, (size_t)cfg->d * 4, s>>>(ra);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return COLIBRI_E_CUDA;
    if (prof_at >= 0 && prof_mark(prof_at, s))
        return COLIBRI_E_CUDA;
    SelectArgs sa{logits, cfg->router == COLIBRI_ROUTER_SOFTMAX ? nullptr : bias, T, cfg->n_exp,
                  cfg->top_k, cfg->n_group, cfg->topk_group, cfg->router, cfg->norm_topk,
                  cfg->routed_scale, ids, w};
    constexpr int SEL_WARPS = 4;
    k_router_select<<<(T + SEL_WARPS - 1) / SEL_WARPS, 32 * SEL_WARPS, 0, s>>>(sa);
    if (cudaGetLastError() != cudaSuccess)
        return COLIBRI_E_CUDA;
    if (prof_at >= 0 && prof_mark(prof_at + 1, s))
        return COLIBRI_E_CUDA;
    return COLIBRI_OK;
}

int colibri_router_topk(const colibri_layer_cfg *cfg, const float *x, int T, const float *Wr,
                        const float *bias, float *logits, int32_t *ids, float *w, void *stream)
{
    if (!cfg_valid(cfg) || T < 0)
        return COLIBRI_E_INVAL;
    if (T == 0)
        return COLIBRI_OK;
    if (!x || !Wr || !logits || !ids || !w || !aligned(Wr, 16))
        return COLIBRI_E_INVAL;
    return launch_router(cfg, x, T, Wr, bias, logits, ids, w, nullptr, (cudaStream_t)stream, -1);
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

    if (prof_mark(0, s))
        return COLIBRI_E_CUDA;
    // a1: q8 of x (plain codes + even/odd codes + corrections); clears the error flag
    Q8Args qa{x, T, d, reinterpret_cast<int8_t *>(ws + L.qx), reinterpret_cast<float *>(ws + L.sx),
              reinterpret_cast<int8_t *>(ws + L.qx_eo), reinterpret_cast<int *>(ws + L.xc), err};
    const long groups = (long)T * (d / G);
    k_q8<<<(unsigned)((groups + 7) / 8), 256, 0, s>>>(qa);
    if (cudaGetLastError() != cudaSuccess || prof_mark(1, s))
        return COLIBRI_E_CUDA;

    // a2-a3: router
    if (!ids_given) {
        int rc = launch_router(cfg, x, T, Wr, bias, reinterpret_cast<float *>(ws + L.logits), ids, w,
                               err, s, g_prof.on ? 2 : -1);
        if (rc)
            return rc;
    } else if (prof_mark(2, s) || prof_mark(3, s)) {
        return COLIBRI_E_CUDA;
    }

    // a4: bucketing and slot list
    const int down_blocks = (d + DN_ROWS - 1) / DN_ROWS;
    BucketArgs ba{ids, T, K, E, cfg->has_shared, cfg->shared_ffn, cfg->ffn, down_blocks,
                  reinterpret_cast<int32_t *>(ws + L.offsets), reinterpret_cast<int32_t *>(ws + L.pairs),
                  reinterpret_cast<Slot *>(ws + L.slots), reinterpret_cast<Counters *>(ws + L.counters), err};
    const size_t bsm = (size_t)34 * E * sizeof(int);
    static bool bucket_attr_set = false;
    if (bsm > 48 * 1024 && !bucket_attr_set) {
        if (cudaFuncSetAttribute(k_bucket, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bsm) !=
            cudaSuccess)
            return COLIBRI_E_CUDA;
        bucket_attr_set = true;
    }
    k_bucket<<<1, 1024, bsm, s>>>(ba);
    if (cudaGetLastError() != cudaSuccess || prof_mark(4, s))
        return COLIBRI_E_CUDA;

    // a6-a8: gate/up (+ SwiGLU + q8 h), then down, for every slot (shared expert first)
    colibri_expert sh{};
    if (cfg->has_shared)
        sh = *shared;
    const int routed_slots = T * K < E ? T * K : E;
    const int gu_items = (cfg->has_shared ? cfg->shared_ffn / G : 0) + routed_slots * (cfg->ffn / G);
    GateUpArgs ga{experts, sh, d, cfg->ffn, cfg->shared_ffn, T, K, cfg->has_shared, (int)L.fmax,
                  reinterpret_cast<const Slot *>(ws + L.slots), reinterpret_cast<const Counters *>(ws + L.counters),
                  reinterpret_cast<const int32_t *>(ws + L.pairs), reinterpret_cast<const int8_t *>(ws + L.qx_eo),
                  reinterpret_cast<const float *>(ws + L.sx), reinterpret_cast<const int *>(ws + L.xc),
                  reinterpret_cast<int8_t *>(ws + L.hq), reinterpret_cast<int8_t *>(ws + L.hq_eo),
                  reinterpret_cast<float *>(ws + L.hs), reinterpret_cast<int *>(ws + L.hc)};
    if (launch_gateup(ga, gu_items, s) != cudaSuccess || prof_mark(5, s))
        return COLIBRI_E_CUDA;
    const int dn_items = (routed_slots + (cfg->has_shared ? 1 : 0)) * down_blocks;
    DownArgs da{experts, sh, d, cfg->ffn, cfg->shared_ffn, T, K, cfg->has_shared, (int)L.fmax,
                reinterpret_cast<const Slot *>(ws + L.slots), reinterpret_cast<const Counters *>(ws + L.counters),
                reinterpret_cast<const int32_t *>(ws + L.pairs), reinterpret_cast<const int8_t *>(ws + L.hq_eo),
                reinterpret_cast<const float *>(ws + L.hs), reinterpret_cast<const int *>(ws + L.hc),
                reinterpret_cast<float *>(ws + L.y)};
    if (launch_down(da, dn_items, s) != cudaSuccess || prof_mark(6, s))
        return COLIBRI_E_CUDA;

    // a9: combine
    CombineArgs ca{reinterpret_cast<const float *>(ws + L.y), w, T, K, d, cfg->has_shared, out};
    dim3 cg((d / 4 + 255) / 256, T);
    k_combine<<<cg, 256, 0, s>>>(ca);
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

int colibri_debug_group_dots(const uint8_t *w, const int8_t *qa, int rows, int cols, int32_t *dots,
                             void *stream)
{
    if (!w || !qa || !dots || rows < 0 || cols <= 0 || cols % G)
        return COLIBRI_E_INVAL;
    if (rows == 0)
        return COLIBRI_OK;
    if (!aligned(w, 16) || !aligned(qa, 16))
        return COLIBRI_E_INVAL;
    k_debug_dots<<<(rows + 7) / 8, 256, 0, (cudaStream_t)stream>>>(w, qa, rows, cols, dots);
    return cuda_status(cudaGetLastError());
}

}  // extern "C"
