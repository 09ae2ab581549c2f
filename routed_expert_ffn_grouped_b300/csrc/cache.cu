// HBM expert cache: an LRU table of blob-sized slots fed from pinned host memory.
//
// The pages describe experts streaming on demand through an LRU cache with
// asynchronous readahead and a lookahead thread that prefetches the next layer's
// experts while the current one computes (dashen-tech guide, bullet "Streaming
// d'experts", "Analyse approfondie" step 2 and section "Router-Lookahead prefetch").
// Here the slow tier is pinned host memory and the readahead is cudaMemcpyAsync on a
// copy stream; the compute stream waits on per-slot events instead of a thread. Demand
// misses and prefetches may use two streams, so that a miss never queues behind a
// speculative copy. Prefetches are either whole-blob copies issued at once, or a queue
// of chunked copies that the host issues only while no demand copy runs (while it waits
// for the layer whose output names the next experts) and that a lookup of their layer
// finishes (named ids) or cancels (the others): a wrong guess then costs at most the
// chunks in flight, not a whole blob.
#include <algorithm>
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
    cudaStream_t pcopy = nullptr;       // prefetch copies (nullptr: the copy stream)
    int max_prefetch = 0;               // prefetch copies (chunks) in flight at most (0: no cap)
    std::vector<int> prefetch_inflight; // slots whose prefetch copy may still be running
    // queued prefetch (chunk_bytes > 0)
    struct Pending {
        int64_t key;
        int slot;
        size_t issued;                  // bytes of the blob already enqueued
    };
    size_t chunk_bytes = 0;
    std::vector<Pending> queue;         // prefetches not fully enqueued, in stage order
    std::vector<char> pending;          // per slot: holds a queued prefetch
    std::vector<cudaEvent_t> chunk_ev;  // ring of the chunks in flight
    int chunk_head = 0, chunks_out = 0;
    cudaEvent_t demand_tail = nullptr;  // after the last demand copy
    bool has_demand = false;
    cudaEvent_t wait_ev = nullptr;
    LruCore lru{1};
    std::vector<cudaEvent_t> ready;     // per slot: its blob (and table entry) has landed
    std::vector<cudaEvent_t> use_done;  // per slot: the compute that read it has finished
    std::vector<char> has_use;          // use_done recorded at least once
    std::vector<char> has_ready;        // ready recorded at least once
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

cudaStream_t prefetch_stream(const colibri_cache *c)
{
    return c->pcopy ? c->pcopy : c->copy;
}

// Orders the next copy into `slot` on stream q after the compute that last read the slot
// and after any earlier copy into it (on either stream: a prefetch evicted or cancelled
// before its first use may still be running).
int order_slot(colibri_cache *c, int slot, cudaStream_t q)
{
    if (c->has_use[slot] && cudaStreamWaitEvent(q, c->use_done[slot], 0) != cudaSuccess)
        return COLIBRI_E_CUDA;
    if (c->has_ready[slot] && cudaStreamWaitEvent(q, c->ready[slot], 0) != cudaSuccess)
        return COLIBRI_E_CUDA;
    return COLIBRI_OK;
}

// Copies bytes [from, nbytes) of blob `key` into `slot` on stream q, then writes the
// table entry and records the slot's ready event.
int stage_into(colibri_cache *c, int64_t key, int slot, cudaStream_t q, size_t from = 0)
{
    if (c->fail_next > 0) {
        --c->fail_next;
        c->lru.erase(key);
        return COLIBRI_E_STAGE;
    }
    if (int rc = order_slot(c, slot, q))
        return rc;
    char *dst = c->slots + (size_t)slot * c->lay.nbytes;
    const char *src = c->host + (size_t)key * c->lay.nbytes;
    if (cudaMemcpyAsync(dst + from, src + from, c->lay.nbytes - from, cudaMemcpyHostToDevice, q) != cudaSuccess)
        return COLIBRI_E_CUDA;
    k_set_entry<<<1, 1, 0, q>>>(c->dtables + key, entry_for(c, slot));
    if (cudaGetLastError() != cudaSuccess)
        return COLIBRI_E_CUDA;
    if (cudaEventRecord(c->ready[slot], q) != cudaSuccess)
        return COLIBRI_E_CUDA;
    c->has_ready[slot] = 1;
    c->st.bytes_staged += (int64_t)(c->lay.nbytes - from);
    return COLIBRI_OK;
}

int queue_index(const colibri_cache *c, int slot)
{
    for (size_t i = 0; i < c->queue.size(); ++i)
        if (c->queue[i].slot == slot)
            return (int)i;
    return -1;
}

// Takes queue entry i out of the queue. Its chunks already enqueued stay ordered before
// any later copy into the slot (its ready event is recorded behind them).
int unqueue(colibri_cache *c, int i)
{
    const colibri_cache::Pending p = c->queue[i];
    c->queue.erase(c->queue.begin() + i);
    c->pending[p.slot] = 0;
    if (p.issued > 0) {
        if (cudaEventRecord(c->ready[p.slot], prefetch_stream(c)) != cudaSuccess)
            return COLIBRI_E_CUDA;
        c->has_ready[p.slot] = 1;
    }
    return COLIBRI_OK;
}

// A slot was taken from `evicted` for another key: a queued prefetch there is cancelled.
int on_evict(colibri_cache *c, int slot, int64_t evicted)
{
    if (evicted < 0)
        return COLIBRI_OK;
    ++c->st.evictions;
    if (!c->pending[slot])
        return COLIBRI_OK;
    ++c->st.prefetch_cancelled;
    return unqueue(c, queue_index(c, slot));
}

// Chunks still in flight, after retiring the finished ones from the ring.
int chunks_in_flight(colibri_cache *c)
{
    while (c->chunks_out > 0) {
        const cudaError_t e = cudaEventQuery(c->chunk_ev[c->chunk_head]);
        if (e == cudaErrorNotReady)
            break;
        if (e != cudaSuccess)
            (void)cudaGetLastError();
        c->chunk_head = (c->chunk_head + 1) % (int)c->chunk_ev.size();
        --c->chunks_out;
    }
    return c->chunks_out;
}

bool chunk_in_flight_any(colibri_cache *c)
{
    return !c->chunk_ev.empty() && chunks_in_flight(c) > 0;
}

// Enqueues up to max_chunks queued prefetch chunks on the prefetch stream while no demand
// copy is running and fewer than the cap are in flight; a blob's last chunk writes its
// table entry. *enqueued counts them.
int pump(colibri_cache *c, int max_chunks, int *enqueued)
{
    *enqueued = 0;
    if (c->queue.empty())
        return COLIBRI_OK;
    if (c->has_demand) {
        const cudaError_t e = cudaEventQuery(c->demand_tail);
        if (e == cudaErrorNotReady)
            return COLIBRI_OK;
        if (e != cudaSuccess)
            return COLIBRI_E_CUDA;
    }
    const cudaStream_t q = prefetch_stream(c);
    while (*enqueued < max_chunks && !c->queue.empty() && chunks_in_flight(c) < (int)c->chunk_ev.size()) {
        colibri_cache::Pending &p = c->queue.front();
        if (p.issued == 0 && order_slot(c, p.slot, q))
            return COLIBRI_E_CUDA;
        const size_t n = std::min(c->chunk_bytes, c->lay.nbytes - p.issued);
        char *dst = c->slots + (size_t)p.slot * c->lay.nbytes + p.issued;
        const char *src = c->host + (size_t)p.key * c->lay.nbytes + p.issued;
        if (cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, q) != cudaSuccess)
            return COLIBRI_E_CUDA;
        const int ring = (int)c->chunk_ev.size();
        if (cudaEventRecord(c->chunk_ev[(c->chunk_head + c->chunks_out) % ring], q) != cudaSuccess)
            return COLIBRI_E_CUDA;
        ++c->chunks_out;
        ++*enqueued;
        p.issued += n;
        c->st.bytes_staged += (int64_t)n;
        c->st.prefetch_bytes += (int64_t)n;
        if (p.issued == c->lay.nbytes) {
            k_set_entry<<<1, 1, 0, q>>>(c->dtables + p.key, entry_for(c, p.slot));
            if (cudaGetLastError() != cudaSuccess)
                return COLIBRI_E_CUDA;
            if (cudaEventRecord(c->ready[p.slot], q) != cudaSuccess)
                return COLIBRI_E_CUDA;
            c->has_ready[p.slot] = 1;
            c->pending[p.slot] = 0;
            c->queue.erase(c->queue.begin());
        }
    }
    return COLIBRI_OK;
}

// A lookup of `layer` settles that layer's queued prefetches: a named id's blob is
// finished on the demand (copy) stream after its chunks so far; the others are cancelled
// and their slots freed.
int settle_layer(colibri_cache *c, int layer, const int32_t *ids, int n)
{
    for (size_t i = 0; i < c->queue.size();) {
        const colibri_cache::Pending p = c->queue[i];
        if (p.key / c->n_exp != layer) {
            ++i;
            continue;
        }
        const int id = (int)(p.key % c->n_exp);
        const bool named = std::find(ids, ids + n, id) != ids + n;
        if (int rc = unqueue(c, (int)i))
            return rc;
        if (named) {
            if (int rc = stage_into(c, p.key, p.slot, c->copy, p.issued))
                return rc;
            c->has_demand = true;
            if (cudaEventRecord(c->demand_tail, c->copy) != cudaSuccess)
                return COLIBRI_E_CUDA;
        } else {
            c->lru.erase(p.key);
            c->prefetched[p.slot] = 0;
            ++c->st.prefetch_cancelled;
        }
    }
    return COLIBRI_OK;
}

// Prefetch copies still running (their slot's ready event not yet reached), after
// dropping the finished ones from the list.
int prefetches_in_flight(colibri_cache *c)
{
    size_t k = 0;
    for (int slot : c->prefetch_inflight) {
        const cudaError_t e = cudaEventQuery(c->ready[slot]);
        if (e == cudaErrorNotReady)
            c->prefetch_inflight[k++] = slot;
        else if (e != cudaSuccess)
            (void)cudaGetLastError();
    }
    c->prefetch_inflight.resize(k);
    return (int)k;
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
    c->has_ready.assign(n_slots, 0);
    c->prefetched.assign(n_slots, 0);
    c->pending.assign(n_slots, 0);
    c->st.n_slots = (int)n_slots;
    bool ok = cudaEventCreateWithFlags(&c->sync_ev, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&c->demand_tail, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&c->wait_ev, cudaEventDisableTiming) == cudaSuccess;
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
        if (c->chunk_bytes == 0 && c->max_prefetch > 0 && !c->lru.contains(key) &&
            prefetches_in_flight(c) >= c->max_prefetch) {
            ++c->st.prefetch_throttled;  // the copy engine is behind: do not queue more
            continue;
        }
        const LruCore::Result r = c->lru.access(key, false, false);  // a prefetch is not a use
        if (r.result == 2) {
            ++c->st.prefetch_skipped;
            continue;
        }
        if (r.result == 1)
            continue;
        if (int rc = on_evict(c, r.slot, r.evicted))
            return rc;
        if (c->chunk_bytes > 0) {
            c->queue.push_back({key, r.slot, 0});
            c->pending[r.slot] = 1;
        } else {
            if (int rc = stage_into(c, key, r.slot, prefetch_stream(c)))
                return rc;
            c->st.prefetch_bytes += (int64_t)c->lay.nbytes;
            c->prefetch_inflight.push_back(r.slot);
        }
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
    if (int rc = settle_layer(c, layer, ids, n))
        return rc;
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
            if (int rc = on_evict(c, r.slot, r.evicted))
                return rc;
            c->prefetched[r.slot] = 0;
            int rc = stage_into(c, key, r.slot, c->copy);
            if (rc)
                return rc;
            c->has_demand = true;
            if (cudaEventRecord(c->demand_tail, c->copy) != cudaSuccess)
                return COLIBRI_E_CUDA;
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

int colibri_expert_cache_set_prefetch(colibri_cache *c, void *prefetch_stream, int max_in_flight,
                                      size_t chunk_bytes)
{
    if (!c || max_in_flight < 0 || (chunk_bytes > 0 && (max_in_flight < 1 || max_in_flight > 64)))
        return COLIBRI_E_INVAL;
    if (!c->queue.empty() || chunk_in_flight_any(c))
        return COLIBRI_E_INVAL;
    DeviceGuard g(c->device);
    for (cudaEvent_t e : c->chunk_ev)
        cudaEventDestroy(e);
    c->chunk_ev.clear();
    c->chunk_head = c->chunks_out = 0;
    if (chunk_bytes > 0) {
        c->chunk_ev.resize(max_in_flight, nullptr);
        for (cudaEvent_t &e : c->chunk_ev)
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
                for (cudaEvent_t x : c->chunk_ev)
                    if (x)
                        cudaEventDestroy(x);
                c->chunk_ev.clear();
                c->chunk_bytes = 0;
                return COLIBRI_E_CUDA;
            }
    }
    c->pcopy = static_cast<cudaStream_t>(prefetch_stream);
    c->max_prefetch = max_in_flight;
    c->chunk_bytes = chunk_bytes;
    return COLIBRI_OK;
}

int colibri_expert_cache_pump(colibri_cache *c, int max_chunks, int *enqueued)
{
    if (!c || max_chunks < 0 || !enqueued)
        return COLIBRI_E_INVAL;
    DeviceGuard g(c->device);
    return pump(c, max_chunks, enqueued);
}

int colibri_expert_cache_wait(colibri_cache *c, void *stream, int timeout_ms)
{
    if (!c || timeout_ms < 0)
        return COLIBRI_E_INVAL;
    DeviceGuard g(c->device);
    if (cudaEventRecord(c->wait_ev, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return COLIBRI_E_CUDA;
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        const cudaError_t e = cudaEventQuery(c->wait_ev);
        if (e == cudaSuccess)
            return COLIBRI_OK;
        if (e != cudaErrorNotReady)
            return COLIBRI_E_CUDA;
        int n = 0;
        if (int rc = pump(c, 1 << 30, &n))
            return rc;
        const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                            std::chrono::steady_clock::now() - t0)
                            .count();
        if (ms >= timeout_ms)
            return COLIBRI_E_TIMEOUT;
        std::this_thread::yield();
    }
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
    if (c->pcopy && c->pcopy != c->copy && cudaStreamWaitEvent(c->pcopy, c->sync_ev, 0) != cudaSuccess)
        return COLIBRI_E_CUDA;
    if (c->pcopy && c->pcopy != c->copy && cudaEventRecord(c->sync_ev, c->pcopy) != cudaSuccess)
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
    for (cudaEvent_t e : c->chunk_ev)
        if (e)
            cudaEventDestroy(e);
    for (cudaEvent_t e : {c->sync_ev, c->demand_tail, c->wait_ev})
        if (e)
            cudaEventDestroy(e);
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
