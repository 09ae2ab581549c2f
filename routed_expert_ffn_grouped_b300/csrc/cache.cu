// HBM expert cache: an LRU table of blob-sized slots fed from pinned host memory.
//
// The pages describe experts streaming on demand through an LRU cache with
// asynchronous readahead and a lookahead thread that prefetches the next layer's
// experts while the current one computes (dashen-tech guide, bullet "Streaming
// d'experts", "Analyse approfondie" step 2 and section "Router-Lookahead prefetch").
// Here the slow tier is pinned host memory and the readahead is cudaMemcpyAsync on a
// copy stream; the compute stream waits on per-slot events instead of a thread.
#include <chrono>
#include <thread>
#include <unordered_map>
#include <vector>

#include "common.cuh"
#include "lru.h"

using clb::LruCore;

struct colibri_cache {
    int device = 0;
    char *pool = nullptr;
    size_t pool_bytes = 0;
    const char *host = nullptr;
    int n_layers = 0, n_exp = 0, d = 0, ffn = 0, top_k = 0;
    colibri_blob_layout lay{};
    colibri_expert *dtables = nullptr;  // [n_layers][n_exp], at the start of the pool
    char *slots = nullptr;
    int n_slots = 0;
    cudaStream_t copy = nullptr;
    LruCore lru{1};
    std::vector<cudaEvent_t> ready;     // per slot: its blob (and table entry) has landed
    std::vector<cudaEvent_t> use_done;  // per slot: the compute that read it has finished
    std::vector<char> has_use;          // use_done recorded at least once
    std::vector<char> prefetched;       // staged by a prefetch and not looked up since
    std::vector<int> pinned_slots;      // slots of the current lookup batch
    cudaEvent_t sync_ev = nullptr;
    int strict = 0;
    int fail_next = 0;
    colibri_cache_stats st{};
};

namespace {

__global__ void k_set_entry(colibri_expert *dst, colibri_expert v)
{
    *dst = v;
}

colibri_expert entry_for(const colibri_cache *c, int slot)
{
    const char *b = c->slots + (size_t)slot * c->lay.nbytes;
    colibri_expert e;
    e.w1 = reinterpret_cast<const uint8_t *>(b + c->lay.w1);
    e.w3 = reinterpret_cast<const uint8_t *>(b + c->lay.w3);
    e.w2 = reinterpret_cast<const uint8_t *>(b + c->lay.w2);
    e.s1 = reinterpret_cast<const float *>(b + c->lay.s1);
    e.s3 = reinterpret_cast<const float *>(b + c->lay.s3);
    e.s2 = reinterpret_cast<const float *>(b + c->lay.s2);
    return e;
}

// Copies blob `key` into `slot` on the copy stream, after the compute that last read the
// slot, then writes the table entry and records the slot's ready event.
int stage_into(colibri_cache *c, int64_t key, int slot)
{
    if (c->fail_next > 0) {
        --c->fail_next;
        c->lru.erase(key);
        return COLIBRI_E_STAGE;
    }
    if (c->has_use[slot] && cudaStreamWaitEvent(c->copy, c->use_done[slot], 0) != cudaSuccess)
        return COLIBRI_E_CUDA;
    char *dst = c->slots + (size_t)slot * c->lay.nbytes;
    const char *src = c->host + (size_t)key * c->lay.nbytes;
    if (cudaMemcpyAsync(dst, src, c->lay.nbytes, cudaMemcpyHostToDevice, c->copy) != cudaSuccess)
        return COLIBRI_E_CUDA;
    k_set_entry<<<1, 1, 0, c->copy>>>(c->dtables + key, entry_for(c, slot));
    if (cudaGetLastError() != cudaSuccess)
        return COLIBRI_E_CUDA;
    if (cudaEventRecord(c->ready[slot], c->copy) != cudaSuccess)
        return COLIBRI_E_CUDA;
    c->st.bytes_staged += (int64_t)c->lay.nbytes;
    return COLIBRI_OK;
}

struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) == cudaSuccess && prev != dev)
            cudaSetDevice(dev);
        else
            prev = -1;
    }
    ~DeviceGuard()
    {
        if (prev >= 0)
            cudaSetDevice(prev);
    }
};

}  // namespace

extern "C" {

int colibri_expert_cache_init(colibri_cache **out, void *hbm_pool, size_t pool_bytes,
                              const void *pinned_host, int n_layers, int n_exp, int d, int ffn,
                              int top_k, void *copy_stream)
{
    if (!out)
        return COLIBRI_E_INVAL;
    *out = nullptr;
    if (!hbm_pool || !pinned_host || n_layers <= 0 || n_exp <= 0 || top_k <= 0 ||
        (reinterpret_cast<uintptr_t>(hbm_pool) & 255))
        return COLIBRI_E_INVAL;
    colibri_blob_layout lay;
    if (colibri_blob_layout_for(d, ffn, &lay) != COLIBRI_OK)
        return COLIBRI_E_INVAL;
    const size_t tables = ((size_t)n_layers * n_exp * sizeof(colibri_expert) + 255) & ~size_t(255);
    if (pool_bytes < tables)
        return COLIBRI_E_NOMEM;
    const size_t n_slots = (pool_bytes - tables) / lay.nbytes;
    if (n_slots < (size_t)top_k)
        return COLIBRI_E_NOMEM;
    colibri_cache *c = new colibri_cache();
    cudaGetDevice(&c->device);
    c->pool = static_cast<char *>(hbm_pool);
    c->pool_bytes = pool_bytes;
    c->host = static_cast<const char *>(pinned_host);
    c->n_layers = n_layers;
    c->n_exp = n_exp;
    c->d = d;
    c->ffn = ffn;
    c->top_k = top_k;
    c->lay = lay;
    c->dtables = reinterpret_cast<colibri_expert *>(c->pool);
    c->slots = c->pool + tables;
    c->n_slots = (int)n_slots;
    c->copy = static_cast<cudaStream_t>(copy_stream);
    c->lru = LruCore((int)n_slots);
    c->ready.resize(n_slots);
    c->use_done.resize(n_slots);
    c->has_use.assign(n_slots, 0);
    c->prefetched.assign(n_slots, 0);
    c->st.n_slots = (int)n_slots;
    bool ok = cudaEventCreateWithFlags(&c->sync_ev, cudaEventDisableTiming) == cudaSuccess;
    for (size_t i = 0; ok && i < n_slots; ++i) {
        ok = cudaEventCreateWithFlags(&c->ready[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&c->use_done[i], cudaEventDisableTiming) == cudaSuccess;
    }
    if (!ok) {
        colibri_expert_cache_destroy(c);
        return COLIBRI_E_CUDA;
    }
    *out = c;
    return COLIBRI_OK;
}

int colibri_expert_cache_stage(colibri_cache *c, int layer, const int32_t *ids, int n)
{
    if (!c || layer < 0 || layer >= c->n_layers || n < 0 || (n > 0 && !ids))
        return COLIBRI_E_INVAL;
    DeviceGuard g(c->device);
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= c->n_exp)
            return COLIBRI_E_INVAL;
        const int64_t key = (int64_t)layer * c->n_exp + ids[i];
        const LruCore::Result r = c->lru.access(key, false, false);  // a prefetch is not a use
        if (r.result == 2) {
            ++c->st.prefetch_skipped;
            continue;
        }
        if (r.result == 1)
            continue;
        if (r.evicted >= 0)
            ++c->st.evictions;
        int rc = stage_into(c, key, r.slot);
        if (rc)
            return rc;
        c->prefetched[r.slot] = 1;
        ++c->st.prefetch_staged;
    }
    return COLIBRI_OK;
}

int colibri_expert_cache_lookup(colibri_cache *c, int layer, const int32_t *ids, int n, void *wait_on)
{
    if (!c || layer < 0 || layer >= c->n_layers || n < 0 || (n > 0 && !ids))
        return COLIBRI_E_INVAL;
    for (int i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= c->n_exp)
            return COLIBRI_E_INVAL;
    DeviceGuard g(c->device);
    cudaStream_t s = static_cast<cudaStream_t>(wait_on);
    // Everything enqueued on `s` so far includes the compute of the previous batch:
    // mark its slots' use as done at this point and unpin them.
    for (int slot : c->pinned_slots) {
        if (cudaEventRecord(c->use_done[slot], s) != cudaSuccess)
            return COLIBRI_E_CUDA;
        c->has_use[slot] = 1;
    }
    c->pinned_slots.clear();
    c->lru.unpin_all();
    if (c->strict) {
        for (int i = 0; i < n; ++i)
            if (!c->lru.contains((int64_t)layer * c->n_exp + ids[i]))
                return COLIBRI_E_MISS;
    }
    for (int i = 0; i < n; ++i) {
        const int64_t key = (int64_t)layer * c->n_exp + ids[i];
        const LruCore::Result r = c->lru.access(key, true);
        ++c->st.lookups;
        if (r.result == 2)
            return COLIBRI_E_NOMEM;
        if (r.result == 1) {
            ++c->st.hits;
            if (c->prefetched[r.slot]) {
                ++c->st.prefetch_used;
                c->prefetched[r.slot] = 0;
            }
        } else {
            ++c->st.misses;
            if (r.evicted >= 0)
                ++c->st.evictions;
            c->prefetched[r.slot] = 0;
            int rc = stage_into(c, key, r.slot);
            if (rc)
                return rc;
        }
        c->pinned_slots.push_back(r.slot);
        if (cudaStreamWaitEvent(s, c->ready[r.slot], 0) != cudaSuccess)
            return COLIBRI_E_CUDA;
    }
    return COLIBRI_OK;
}

const colibri_expert *colibri_expert_cache_table(colibri_cache *c, int layer)
{
    if (!c || layer < 0 || layer >= c->n_layers)
        return nullptr;
    return c->dtables + (size_t)layer * c->n_exp;
}

int colibri_expert_cache_set_hot(colibri_cache *c, int n_hot)
{
    if (!c || n_hot < 0 || n_hot > c->n_slots - c->top_k)
        return COLIBRI_E_INVAL;
    c->lru.set_hot(n_hot);
    return COLIBRI_OK;
}

int colibri_expert_cache_set_strict(colibri_cache *c, int strict)
{
    if (!c)
        return COLIBRI_E_INVAL;
    c->strict = strict ? 1 : 0;
    return COLIBRI_OK;
}

int colibri_expert_cache_stats(colibri_cache *c, colibri_cache_stats *out)
{
    if (!c || !out)
        return COLIBRI_E_INVAL;
    *out = c->st;
    return COLIBRI_OK;
}

int colibri_expert_cache_sync(colibri_cache *c, int timeout_ms)
{
    if (!c)
        return COLIBRI_E_INVAL;
    DeviceGuard g(c->device);
    if (cudaEventRecord(c->sync_ev, c->copy) != cudaSuccess)
        return COLIBRI_E_CUDA;
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        const cudaError_t e = cudaEventQuery(c->sync_ev);
        if (e == cudaSuccess)
            return COLIBRI_OK;
        if (e != cudaErrorNotReady)
            return COLIBRI_E_CUDA;
        const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                            std::chrono::steady_clock::now() - t0)
                            .count();
        if (ms >= timeout_ms)
            return COLIBRI_E_TIMEOUT;
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
}

void colibri_expert_cache_destroy(colibri_cache *c)
{
    if (!c)
        return;
    DeviceGuard g(c->device);
    for (cudaEvent_t e : c->ready)
        if (e)
            cudaEventDestroy(e);
    for (cudaEvent_t e : c->use_done)
        if (e)
            cudaEventDestroy(e);
    if (c->sync_ev)
        cudaEventDestroy(c->sync_ev);
    delete c;
}

int colibri_expert_cache_inject_stage_failure(colibri_cache *c, int count)
{
    if (!c || count < 0)
        return COLIBRI_E_INVAL;
    c->fail_next = count;
    return COLIBRI_OK;
}

int colibri_lru_trace(int capacity, int64_t n_ops, const int32_t *kind, const int64_t *key, int8_t *result)
{
    return colibri_lru_trace_hot(capacity, 0, n_ops, kind, key, result);
}

int colibri_lru_trace_hot(int capacity, int n_hot, int64_t n_ops, const int32_t *kind, const int64_t *key,
                          int8_t *result)
{
    if (capacity <= 0 || n_hot < 0 || n_hot > capacity || n_ops < 0 || (n_ops > 0 && (!kind || !key || !result)))
        return COLIBRI_E_INVAL;
    LruCore lru(capacity, n_hot);
    for (int64_t i = 0; i < n_ops; ++i) {
        if (kind[i] == 0) {
            lru.unpin_all();
            result[i] = 0;
        } else if (kind[i] == 1 || kind[i] == 2) {
            result[i] = (int8_t)lru.access(key[i], kind[i] == 1, kind[i] == 1).result;
        } else {
            return COLIBRI_E_INVAL;
        }
    }
    return COLIBRI_OK;
}

}  // extern "C"
