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

#include "colibri.h"

namespace {

// The workspace of every call of colibri_moe_layer_noalloc. A __device__ array lives in
// each device's memory from the moment the library's module is loaded on that device
// until the process exits. Host code must not take its address with `&`: on the host
// the name stands for a host-side shadow, not for device memory. The device address
// comes from cudaGetSymbolAddress, once per device (see scratch_for_current_device).
static __device__ __align__(256) unsigned char g_noalloc_scratch[COLIBRI_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on the first
// call made with that device current. Returns nullptr if the lookup fails.
void *scratch_for_current_device(int *status)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *status = COLIBRI_E_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            *status = COLIBRI_E_CUDA;
            return nullptr;
        }
        g_ptr[dev] = p;
    }
    *status = COLIBRI_OK;
    return g_ptr[dev];
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
    // The layer clears the scratch's error flag in its first kernel and writes every other
    // intermediate before reading it, so nothing left from an earlier call leaks through.
    return colibri_moe_layer(cfg, x, T, Wr, bias, experts, shared, ids, w, ids_given, out, ws,
                             (size_t)COLIBRI_NOALLOC_SCRATCH_BYTES, stream);
}
