// colibri_moe_layer_noalloc: the layer of colibri_moe_layer with its workspace taken
// from a fixed array that the library itself holds in device memory, so that the caller
// never has to allocate one.
//
// Some callers cannot allocate device memory at the moment they run the layer: a host
// runtime that hands out all device memory through its own pool and forbids other
// allocations once it has started, a plugin that is given only input and output
// buffers, or a latency-critical loop where cudaMalloc's implicit synchronisation of the
// device would stall every other stream. This entry point serves them.
#include <mutex>

#include <cuda.h>

#include "colibri.h"

namespace {

// The workspace of every call of colibri_moe_layer_noalloc. A __device__ array lives in
// each device's memory from the moment the library's module is loaded on that device
// until the process exits. Host code must not take its address with `&`: on the host
// the name stands for a host-side shadow, not for device memory. The device address
// comes from cudaGetSymbolAddress (see scratch_for_current_device).
static __device__ __align__(256) unsigned char g_noalloc_scratch[COLIBRI_NOALLOC_SCRATCH_BYTES];

// The array's address on each device, with the id of the context it was looked up in.
// A context that is destroyed and created again (cudaDeviceReset, or the primary context
// released and retained anew) loads the module again, possibly at another address; its
// id differs from every earlier context's, so the address is looked up again.
constexpr int kMaxDevices = 64;
struct Cached {
    unsigned long long ctx_id;
    void *ptr;
};
std::mutex g_mu;
Cached g_cache[kMaxDevices] = {};

// Driver entry points, resolved through the runtime (the library does not link libcuda).
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;

bool resolve_driver_calls()
{
    if (g_ctx_current && g_ctx_id)
        return true;
    void *a = nullptr, *b = nullptr;
    cudaDriverEntryPointQueryResult qa{}, qb{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) != cudaSuccess ||
        qa != cudaDriverEntryPointSuccess || qb != cudaDriverEntryPointSuccess || !a || !b)
        return false;
    g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(a);
    g_ctx_id = reinterpret_cast<CtxGetIdFn>(b);
    return true;
}

// Id of the calling thread's current context, or 0 when none is current yet.
unsigned long long current_ctx_id()
{
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx || g_ctx_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array in the current device's context. The set-up (the
// cudaGetSymbolAddress lookup, which also loads the library's module in that context if
// it is not loaded yet) runs on the first call made in each context, including the first
// call after a device reset. Returns nullptr, with *status set, if a lookup fails.
void *scratch_for_current_device(int *status)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *status = COLIBRI_E_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!resolve_driver_calls()) {
        *status = COLIBRI_E_CUDA;
        return nullptr;
    }
    const unsigned long long id = current_ctx_id();
    if (id == 0 || g_cache[dev].ctx_id != id || !g_cache[dev].ptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            *status = COLIBRI_E_CUDA;
            return nullptr;
        }
        // the lookup made the device's primary context current if none was
        const unsigned long long now = current_ctx_id();
        g_cache[dev].ctx_id = now;
        g_cache[dev].ptr = now ? p : nullptr;
        *status = COLIBRI_OK;
        return p;
    }
    *status = COLIBRI_OK;
    return g_cache[dev].ptr;
}

}  // namespace

extern "C" int colibri_moe_layer_noalloc(const colibri_layer_cfg *cfg, const float *x, int T,
                                         const float *Wr, const float *bias,
                                         const colibri_expert *experts, const colibri_expert *shared,
                                         int32_t *ids, float *w, int ids_given, float *out,
                                         void *stream)
{
    const size_t need = colibri_moe_workspace_bytes(cfg, T < 0 ? 0 : T);
    if (need == 0 || T < 0)
        return COLIBRI_E_INVAL;
    if (need > (size_t)COLIBRI_NOALLOC_SCRATCH_BYTES)
        return COLIBRI_E_NOMEM;
    if (T == 0)
        return COLIBRI_OK;
    int st = COLIBRI_OK;
    void *ws = scratch_for_current_device(&st);
    if (!ws)
        return st;
    // colibri_moe_layer's host code clears the scratch's error flag and the kernels' sync
    // counters with a memset on the stream before its first kernel, and the kernels write
    // every other intermediate before reading it, so nothing left from an earlier call
    // leaks through.
    return colibri_moe_layer(cfg, x, T, Wr, bias, experts, shared, ids, w, ids_given, out, ws,
                             (size_t)COLIBRI_NOALLOC_SCRATCH_BYTES, stream);
}
