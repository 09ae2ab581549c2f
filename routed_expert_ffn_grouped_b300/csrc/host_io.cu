// colibri_moe_layer_host: one blocking call of the layer on host buffers. It copies the
// step's activations (and given ids and weights) from host memory into a device region
// at the end of the workspace, runs colibri_moe_layer there, and copies the output, the
// routing results and the device error flag back, all on one stream, then waits for it.
//
// This serves a host runtime that keeps its activations in host memory between layers
// (the hybrid CPU/GPU setting of the Colibri pages, "Streaming d'experts" in "Guide
// Complet de Colibri"): a whole step is one C call, with no per-copy round trip through
// the caller.
#include "colibri.h"
#include "workspace.h"

namespace {

// A page-locked word per host thread for the device error flag, so that its copy back is
// an ordinary asynchronous copy on the stream (allocated on the thread's first call, kept
// until the thread exits).
struct PinnedFlag {
    int *p = nullptr;
    ~PinnedFlag()
    {
        if (p)
            cudaFreeHost(p);
    }
};
thread_local PinnedFlag t_flag;

size_t up256(size_t n)
{
    return (n + 255) & ~size_t(255);
}

// Offsets of the device copies of the host buffers, after the layer's own workspace.
struct HostIo {
    size_t layer, x, out, ids, w, total;
};

HostIo host_io(const colibri_layer_cfg *c, int T)
{
    HostIo h{};
    const size_t xb = 4 * (size_t)T * c->d, kb = 4 * (size_t)T * c->top_k;
    h.layer = clb::ws_layout(c, T).total;  // 256-byte multiple
    h.x = h.layer;
    h.out = up256(h.x + xb);
    h.ids = up256(h.out + xb);
    h.w = up256(h.ids + kb);
    h.total = up256(h.w + kb);
    return h;
}

bool aligned(const void *p, size_t a)
{
    return (reinterpret_cast<size_t>(p) & (a - 1)) == 0;
}

}  // namespace

extern "C" size_t colibri_moe_host_workspace_bytes(const colibri_layer_cfg *cfg, int T_max)
{
    if (!clb::cfg_valid(cfg) || T_max < 0)
        return 0;
    return host_io(cfg, T_max).total;
}

extern "C" int colibri_moe_layer_host(const colibri_layer_cfg *cfg, const float *x, int T,
                                      const float *Wr, const float *bias,
                                      const colibri_expert *experts, const colibri_expert *shared,
                                      int32_t *ids, float *w, int ids_given, float *out,
                                      void *workspace, size_t ws_bytes, void *stream)
{
    if (!clb::cfg_valid(cfg) || T < 0)
        return COLIBRI_E_INVAL;
    if (T == 0)
        return COLIBRI_OK;
    if (!x || !out || !workspace || !aligned(workspace, 256))
        return COLIBRI_E_INVAL;
    if (ids_given && (!ids || !w))
        return COLIBRI_E_INVAL;
    const HostIo io = host_io(cfg, T);
    if (ws_bytes < io.total)
        return COLIBRI_E_NOMEM;
    cudaStream_t s = (cudaStream_t)stream;
    char *ws = static_cast<char *>(workspace);
    float *dx = reinterpret_cast<float *>(ws + io.x);
    float *dout = reinterpret_cast<float *>(ws + io.out);
    int32_t *dids = reinterpret_cast<int32_t *>(ws + io.ids);
    float *dw = reinterpret_cast<float *>(ws + io.w);
    const size_t xb = 4 * (size_t)T * cfg->d, kb = 4 * (size_t)T * cfg->top_k;

    int st = COLIBRI_OK;
    if (cudaMemcpyAsync(dx, x, xb, cudaMemcpyHostToDevice, s) != cudaSuccess)
        st = COLIBRI_E_CUDA;
    if (st == COLIBRI_OK && ids_given &&
        (cudaMemcpyAsync(dids, ids, kb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
         cudaMemcpyAsync(dw, w, kb, cudaMemcpyHostToDevice, s) != cudaSuccess))
        st = COLIBRI_E_CUDA;
    if (st == COLIBRI_OK)
        st = colibri_moe_layer(cfg, dx, T, Wr, bias, experts, shared, dids, dw, ids_given, dout, workspace,
                               io.layer, stream);
    if (st != COLIBRI_OK) {
        // copies already queued still read the caller's host buffers: let them finish
        cudaStreamSynchronize(s);
        return st;
    }
    int stack_flag = 0;
    if (!t_flag.p && cudaHostAlloc(reinterpret_cast<void **>(&t_flag.p), sizeof(int), cudaHostAllocDefault) != cudaSuccess) {
        (void)cudaGetLastError();
        t_flag.p = nullptr;
    }
    int *flag = t_flag.p ? t_flag.p : &stack_flag;
    const size_t err_off = clb::ws_layout(cfg, T).err;
    if (cudaMemcpyAsync(out, dout, xb, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        st = COLIBRI_E_CUDA;
    if (st == COLIBRI_OK && !ids_given && ids &&
        cudaMemcpyAsync(ids, dids, kb, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        st = COLIBRI_E_CUDA;
    if (st == COLIBRI_OK && !ids_given && w && cudaMemcpyAsync(w, dw, kb, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        st = COLIBRI_E_CUDA;
    if (st == COLIBRI_OK &&
        cudaMemcpyAsync(flag, ws + err_off, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        st = COLIBRI_E_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return COLIBRI_E_CUDA;
    if (st != COLIBRI_OK)
        return st;
    return *flag ? COLIBRI_E_DEVICE : COLIBRI_OK;
}
