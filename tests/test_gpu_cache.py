"""The HBM expert cache on the GPU, through the C ABI: blobs staged from pinned host
memory land byte for byte, lookups follow the host LRU model, a layer computed through
the cache's expert table equals the same layer on fully resident experts bit for bit,
and failures surface as status codes (strict misses, injected staging failures)."""
import ctypes

import numpy as np
import pytest

from routed_expert_ffn_grouped_b300 import synth

pytestmark = pytest.mark.gpu

SPEC = synth.TINY
N_LAYERS = 3


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from routed_expert_ffn_grouped_b300 import build
    build.build()
    return torch


@pytest.fixture(scope="module")
def C(torch_cuda):
    from routed_expert_ffn_grouped_b300 import colibri
    colibri.lib()
    return colibri


@pytest.fixture(scope="module")
def host(torch_cuda):
    """N_LAYERS tiny layers: blobs in pinned host memory (layer-major), plus the layers."""
    torch = torch_cuda
    layers = [synth.make_layer(SPEC, 0, layer=l) for l in range(N_LAYERS)]
    nb = layers[0].blobs.shape[1]
    pinned = torch.empty((N_LAYERS * SPEC.n_exp, nb), dtype=torch.uint8).pin_memory()
    for l, lay in enumerate(layers):
        pinned[l * SPEC.n_exp:(l + 1) * SPEC.n_exp].copy_(torch.from_numpy(lay.blobs))
    return layers, pinned, nb


def make_cache(torch, C, pinned, n_slots, copy_stream):
    tables = (N_LAYERS * SPEC.n_exp * ctypes.sizeof(C.Expert) + 255) // 256 * 256
    nb = pinned.shape[1]
    pool = torch.empty(tables + n_slots * nb, dtype=torch.uint8, device="cuda")
    cache = C.ExpertCache(pool, pinned, N_LAYERS, SPEC.n_exp, SPEC.d, SPEC.ffn, SPEC.top_k, copy_stream)
    return cache, pool


def raw_bytes(ptr, n):
    """n bytes of device memory at a raw address, copied to the host."""
    import torch

    class Raw:
        def __init__(self, p, n):
            self.__cuda_array_interface__ = {"shape": (n,), "typestr": "|u1", "data": (p, False), "version": 3}
    return torch.as_tensor(Raw(ptr, n), device="cuda").cpu().numpy()


def table_entries(torch, C, cache, layer):
    """The device table of `layer` as host colibri_expert structs."""
    torch.cuda.synchronize()
    raw = raw_bytes(cache.table(layer), SPEC.n_exp * ctypes.sizeof(C.Expert))
    return (C.Expert * SPEC.n_exp).from_buffer_copy(raw.tobytes())


def test_staged_blobs_land_byte_for_byte(torch_cuda, C, host):
    torch = torch_cuda
    layers, pinned, nb = host
    copy = torch.cuda.Stream()
    cache, _ = make_cache(torch, C, pinned, 8, copy)
    ids = np.array([3, 7, 11, 0], np.int32)
    cache.lookup(1, ids, wait_on=torch.cuda.current_stream())
    torch.cuda.synchronize()
    lay = synth.blob_layout(SPEC.d, SPEC.ffn)
    tab = table_entries(torch, C, cache, 1)
    for e in ids:
        base = tab[e].w1 - lay.w1
        got = raw_bytes(base, nb)
        assert np.array_equal(got, layers[1].blobs[e]), f"expert {e}"
        assert tab[e].s2 - tab[e].w1 == lay.s2 - lay.w1
    st = cache.stats()
    assert st["misses"] == 4 and st["hits"] == 0 and st["bytes_staged"] == 4 * nb
    cache.close()


@pytest.mark.parametrize("mode", ["copy_stream", "prefetch_stream", "queued"])
def test_layer_through_cache_equals_resident_layer(torch_cuda, C, host, mode):
    """Decode steps with correlated routing over a cache smaller than the expert set:
    the layer reads its experts through the cache's table and must give the same bits
    as the same layer on fully resident experts. Prefetches go on the copy stream, on a
    stream of their own, or as queued chunks that the host enqueues while it waits for
    the previous layer."""
    torch = torch_cuda
    layers, pinned, nb = host
    copy = torch.cuda.Stream()
    cache, _ = make_cache(torch, C, pinned, 6, copy)        # 6 slots for 3 x 16 experts
    pcopy = torch.cuda.Stream()
    if mode == "prefetch_stream":
        cache.set_prefetch(pcopy, 1)
    elif mode == "queued":
        cache.set_prefetch(pcopy, 2, 16384)
    resident = [C.DeviceLayer(lay) for lay in layers]
    T, steps = 1, 6
    ids_all, w_all = synth.streaming_ids(SPEC.replace(n_exp=SPEC.n_exp), 3, N_LAYERS, steps)
    cfg = C.layer_cfg(SPEC)
    ws = torch.empty(C.colibri_moe_workspace_bytes(cfg, T), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for s in range(steps):
        for l in range(N_LAYERS):
            x = torch.from_numpy(synth.activations(SPEC, s, T, step=l)).cuda()
            ids = torch.from_numpy(ids_all[s, l][None].copy()).cuda()
            w = torch.from_numpy(w_all[s, l][None].copy()).cuda()
            if mode == "queued":
                torch.cuda._sleep(2_000_000)                    # a busy stream to wait on
                cache.wait(stream, 10000)
            cache.lookup(l, ids_all[s, l], wait_on=stream)
            if l + 1 < N_LAYERS and s > 0:
                cache.stage(l + 1, ids_all[s - 1, l + 1])       # next-layer prefetch
            out_c = torch.empty((T, SPEC.d), dtype=torch.float32, device="cuda")
            C.colibri_moe_layer(cfg, x, None, None, cache.table(l), resident[l].shared, ids, w, True, out_c, ws,
                                stream=stream)
            out_r = torch.empty_like(out_c)
            C.colibri_moe_layer(cfg, x, None, None, resident[l].table, resident[l].shared, ids, w, True, out_r,
                                ws, stream=stream)
            torch.cuda.synchronize()
            assert np.array_equal(out_c.cpu().numpy().view(np.uint32), out_r.cpu().numpy().view(np.uint32)), (s, l)
    cache.sync()
    st = cache.stats()
    assert st["hits"] + st["misses"] == st["lookups"] == steps * N_LAYERS * SPEC.top_k
    if mode == "queued":
        assert st["misses"] * nb <= st["bytes_staged"] <= (st["misses"] + st["prefetch_staged"]) * nb
        assert st["prefetch_bytes"] > 0
    else:
        assert st["bytes_staged"] == (st["misses"] + st["prefetch_staged"]) * nb
        assert st["prefetch_bytes"] == st["prefetch_staged"] * nb
    assert st["evictions"] > 0
    cache.close()


def test_queued_prefetch_finishes_named_and_cancels_the_rest(torch_cuda, C, host):
    """Queued, chunked prefetches: the next lookup of their layer finishes the named blobs
    on the demand stream, from where their chunks stopped, and cancels the others (their
    slots freed); blobs that finished before the lookup stay resident. The named blobs
    land byte for byte."""
    torch = torch_cuda
    layers, pinned, nb = host
    copy, pcopy = torch.cuda.Stream(), torch.cuda.Stream()
    cache, _ = make_cache(torch, C, pinned, 12, copy)
    chunk = 16384
    cache.set_prefetch(pcopy, 8, chunk)
    stream = torch.cuda.current_stream()
    lay = synth.blob_layout(SPEC.d, SPEC.ffn)
    per_blob = -(-nb // chunk)
    # layer 1: guesses 1, 2 right and 3, 9, 10 wrong; blob 1 finishes, blob 2 gets 3 chunks
    cache.stage(1, np.array([1, 2, 3, 9, 10], np.int32))
    st = cache.stats()
    assert st["prefetch_staged"] == 5 and st["prefetch_bytes"] == 0 and st["bytes_staged"] == 0
    sent = 0
    while sent < per_blob + 3:
        sent += cache.pump(per_blob + 3 - sent)
        pcopy.synchronize()
    assert cache.stats()["prefetch_bytes"] == nb + 3 * chunk
    named = np.array([1, 2, 5, 6], np.int32)
    cache.lookup(1, named, wait_on=stream)
    torch.cuda.synchronize()
    cache.sync(5000)
    st = cache.stats()
    assert st["prefetch_cancelled"] == 3 and st["prefetch_used"] == 2
    assert st["misses"] == 2 and st["hits"] == 2
    assert st["bytes_staged"] == 4 * nb                     # 1 + 2 (finished) + 5 + 6
    tab = table_entries(torch, C, cache, 1)
    for e in named:
        assert np.array_equal(raw_bytes(tab[e].w1 - lay.w1, nb), layers[1].blobs[e]), f"expert {e}"
    # the cancelled guesses left the cache: looking them up misses
    before = cache.stats()["misses"]
    cache.lookup(1, np.array([3, 9, 10, 1], np.int32), wait_on=stream)
    assert cache.stats()["misses"] - before == 3
    # a wait on a busy stream sends the queue out; a blob that finished stays resident
    cache.stage(2, np.array([4, 7], np.int32))
    torch.cuda._sleep(80_000_000)                           # tens of ms of a busy stream
    cache.wait(stream, 10000)
    pcopy.synchronize()
    st = cache.stats()
    assert st["prefetch_bytes"] == nb + 3 * chunk + 2 * nb
    cache.lookup(2, np.array([4, 0, 1, 2], np.int32), wait_on=stream)
    st2 = cache.stats()
    assert st2["prefetch_cancelled"] == 3 and st2["prefetch_used"] == 3
    torch.cuda.synchronize()
    tab = table_entries(torch, C, cache, 2)
    assert np.array_equal(raw_bytes(tab[4].w1 - lay.w1, nb), layers[2].blobs[4])
    cache.close()


def test_queued_prefetch_evicted_before_use(torch_cuda, C, host):
    """A queued prefetch whose slot a demand miss takes is cancelled; copies into the slot
    stay ordered after the chunks already sent, so both layers' blobs land intact."""
    torch = torch_cuda
    layers, pinned, nb = host
    copy, pcopy = torch.cuda.Stream(), torch.cuda.Stream()
    cache, _ = make_cache(torch, C, pinned, SPEC.top_k + 1, copy)
    chunk = 8192
    cache.set_prefetch(pcopy, 4, chunk)
    stream = torch.cuda.current_stream()
    lay = synth.blob_layout(SPEC.d, SPEC.ffn)
    cache.stage(2, np.arange(SPEC.top_k + 1, dtype=np.int32))   # fills every slot
    assert cache.pump(4) == 4                                   # part of the first blob
    first = np.array([0, 1, 2, 3], np.int32)
    with torch.cuda.stream(copy):
        torch.cuda._sleep(20_000_000)                           # holds the demand copies back a while
    cache.lookup(0, first, wait_on=stream)                      # four misses evict four pending prefetches
    assert cache.pump(4) == 0                                   # demand copies pending: no chunk goes out
    torch.cuda.synchronize()
    cache.sync(5000)
    st = cache.stats()
    assert st["prefetch_cancelled"] == SPEC.top_k and st["misses"] == SPEC.top_k
    assert st["prefetch_bytes"] == 4 * chunk
    tab = table_entries(torch, C, cache, 0)
    for e in first:
        assert np.array_equal(raw_bytes(tab[e].w1 - lay.w1, nb), layers[0].blobs[e]), f"layer 0 expert {e}"
    second = np.array([SPEC.top_k, 5, 6, 7], np.int32)          # the surviving guess is named
    cache.lookup(2, second, wait_on=stream)
    torch.cuda.synchronize()
    cache.sync(5000)
    st = cache.stats()
    assert st["prefetch_used"] == 1
    tab = table_entries(torch, C, cache, 2)
    for e in second:
        assert np.array_equal(raw_bytes(tab[e].w1 - lay.w1, nb), layers[2].blobs[e]), f"layer 2 expert {e}"
    cache.close()


def test_lookups_follow_the_lru_model(torch_cuda, C, orc, host):
    torch = torch_cuda
    _, pinned, _ = host
    copy = torch.cuda.Stream()
    n_slots = 6
    cache, _ = make_cache(torch, C, pinned, n_slots, copy)
    rng = np.random.default_rng(4)
    kinds, keys = [], []
    hits = 0
    for step in range(40):
        layer = int(rng.integers(0, N_LAYERS))
        ids = rng.choice(SPEC.n_exp, size=SPEC.top_k, replace=False).astype(np.int32)
        before = cache.stats()["hits"]
        cache.lookup(layer, ids, wait_on=torch.cuda.current_stream())
        hits += cache.stats()["hits"] - before
        kinds += [0] + [1] * len(ids)
        keys += [0] + [layer * SPEC.n_exp + int(e) for e in ids]
    torch.cuda.synchronize()
    res = orc.lru_trace(n_slots, np.array(kinds, np.int32), np.array(keys, np.int64))
    assert hits == int((res[np.array(kinds) == 1] == 1).sum())
    cache.close()


def test_strict_miss_and_injected_stage_failure(torch_cuda, C, host):
    torch = torch_cuda
    _, pinned, _ = host
    copy = torch.cuda.Stream()
    cache, _ = make_cache(torch, C, pinned, 6, copy)
    cache.set_strict(True)
    with pytest.raises(C.ColibriError) as e:
        cache.lookup(0, np.array([1, 2, 3, 4], np.int32), wait_on=torch.cuda.current_stream())
    assert e.value.status == C.E_MISS
    cache.set_strict(False)
    cache.inject_stage_failure(1)
    with pytest.raises(C.ColibriError) as e:
        cache.lookup(0, np.array([1, 2, 3, 4], np.int32), wait_on=torch.cuda.current_stream())
    assert e.value.status == C.E_STAGE
    # the next lookup works again
    cache.lookup(0, np.array([1, 2, 3, 4], np.int32), wait_on=torch.cuda.current_stream())
    cache.sync(5000)
    torch.cuda.synchronize()
    cache.close()


def test_hot_slots_follow_the_policy(torch_cuda, C, orc, host):
    """With usage-pinned slots the cache's hits are those of the oracle's policy, and a
    hot-set size that would leave no room for a lookup batch is rejected."""
    torch = torch_cuda
    _, pinned, _ = host
    copy = torch.cuda.Stream()
    n_slots = 6
    cache, _ = make_cache(torch, C, pinned, n_slots, copy)
    with pytest.raises(C.ColibriError) as e:
        cache.set_hot(n_slots - SPEC.top_k + 1)
    assert e.value.status == C.E_INVAL
    cache.set_hot(2)
    batches = [[0, 1, 2, 3]] * 3 + [[4, 5, 6, 7], [8, 9, 10, 11], [12, 13, 14, 15], [0, 1, 2, 3]]
    stream = torch.cuda.current_stream()
    kinds, keys = [], []
    before = cache.stats()["hits"]
    for b in batches:
        cache.lookup(0, np.array(b, np.int32), wait_on=stream)
        kinds += [0] + [1] * len(b)
        keys += [0] + list(b)
    torch.cuda.synchronize()
    res = orc.lru_hot_trace(n_slots, 2, np.array(kinds, np.int32), np.array(keys, np.int64))
    assert cache.stats()["hits"] - before == int((res == 1).sum())
    assert res[-4:].tolist() == [1, 1, 0, 0]      # the two hot experts survived the scan
    cache.sync(5000)
    cache.close()
