"""Host-side checks of libcolibri.so: it loads without a GPU, exports every symbol that
include/colibri.h declares, and its host-only logic (blob layout, argument checks, the
cache's LRU policy) agrees with the generator and the oracle. No kernel is launched."""
import ctypes
import os
import re

import numpy as np
import pytest

from routed_expert_ffn_grouped_b300 import build as cbuild
from routed_expert_ffn_grouped_b300 import colibri as C
from routed_expert_ffn_grouped_b300 import synth

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "colibri.h")


@pytest.fixture(scope="module")
def lib():
    cbuild.build()
    return C.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(colibri_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(C.SIGNATURES) == names


def test_blob_layout_matches_generator(lib):
    for spec in (synth.TINY, synth.OLMOE, synth.GLM52):
        a = C.colibri_blob_layout_for(spec.d, spec.ffn)
        b = synth.blob_layout(spec.d, spec.ffn)
        assert (a.w1, a.w3, a.w2, a.s1, a.s3, a.s2, a.nbytes) == (b.w1, b.w3, b.w2, b.s1, b.s3, b.s2, b.nbytes)
    with pytest.raises(C.ColibriError):
        C.colibri_blob_layout_for(100, 64)


def test_strerror(lib):
    assert C.strerror(0) == "ok"
    assert "invalid" in C.strerror(C.E_INVAL)


def test_workspace_bytes_and_config_checks(lib):
    for spec in (synth.TINY, synth.OLMOE, synth.GLM52):
        cfg = C.layer_cfg(spec)
        assert C.colibri_moe_workspace_bytes(cfg, 4) > 0
        assert C.colibri_moe_workspace_bytes(cfg, 2048) > C.colibri_moe_workspace_bytes(cfg, 4)
        assert C.colibri_moe_f32_workspace_bytes(cfg, 32) > C.colibri_moe_f32_workspace_bytes(cfg, 1) > 0
        assert lib.colibri_moe_f32_workspace_bytes(ctypes.byref(cfg), 33) == 0   # decode sizes only
        for T in (1, 4, 32, 33, 2048):
            # the host entry's workspace: the layer's, then room for x, out, ids and w
            extra = C.colibri_moe_host_workspace_bytes(cfg, T) - C.colibri_moe_workspace_bytes(cfg, T)
            assert extra >= 2 * 4 * T * spec.d + 2 * 4 * T * spec.top_k
            assert extra < 2 * 4 * T * spec.d + 2 * 4 * T * spec.top_k + 4 * 256
    bad = C.layer_cfg(synth.TINY.replace(n_group=3))
    assert lib.colibri_moe_workspace_bytes(ctypes.byref(bad), 4) == 0
    assert lib.colibri_moe_host_workspace_bytes(ctypes.byref(bad), 4) == 0
    # 64-element groups are accepted; other group sizes, or shapes that are not multiples
    # of the group, are not
    g64 = C.layer_cfg(synth.TINY)
    g64.group = 64
    assert lib.colibri_moe_workspace_bytes(ctypes.byref(g64), 4) > 0
    for group in (16, 48, 128, 0):
        bad = C.layer_cfg(synth.TINY)
        bad.group = group
        assert lib.colibri_moe_workspace_bytes(ctypes.byref(bad), 4) == 0, group
    bad = C.layer_cfg(synth.TINY.replace(d=96, ffn=64, shared_ffn=64))
    assert lib.colibri_moe_workspace_bytes(ctypes.byref(bad), 4) > 0          # fine at 32
    bad.group = 64
    assert lib.colibri_moe_workspace_bytes(ctypes.byref(bad), 4) == 0         # d = 96 is not a multiple of 64
    # the blob layout per group: same nibbles, half the scale bytes at 64
    l32, l64 = C.colibri_blob_layout_for(512, 256), C.colibri_blob_layout_for(512, 256, 64)
    assert (l64.w1, l64.w3, l64.w2, l64.s1) == (l32.w1, l32.w3, l32.w2, l32.s1)
    assert l64.nbytes - l64.s1 == (l32.nbytes - l32.s1) // 2
    lay = C.BlobLayout()
    assert lib.colibri_blob_layout_for_g(96, 64, 64, ctypes.byref(lay)) == C.E_INVAL
    assert lib.colibri_blob_layout_for_g(512, 256, 48, ctypes.byref(lay)) == C.E_INVAL


def test_argument_errors_detected_on_host(lib):
    # Rejected before anything is enqueued: no device is touched.
    assert lib.colibri_q8_quantize(None, 1, 33, None, None, None) == C.E_INVAL
    assert lib.colibri_q8_quantize(None, 0, 64, None, None, None) == C.OK   # empty is a no-op
    assert lib.colibri_q8_quantize_g(None, 1, 96, 64, None, None, None) == C.E_INVAL
    assert lib.colibri_q8_quantize_g(None, 1, 128, 48, None, None, None) == C.E_INVAL
    assert lib.colibri_q8_quantize_g(None, 0, 128, 64, None, None, None) == C.OK
    cfg = C.layer_cfg(synth.TINY)
    assert lib.colibri_moe_layer(ctypes.byref(cfg), None, 0, None, None, None, None, None, None, 0,
                                 None, None, 0, None) == C.OK
    assert lib.colibri_moe_layer(ctypes.byref(cfg), None, 4, None, None, None, None, None, None, 0,
                                 None, None, 0, None) == C.E_INVAL
    assert lib.colibri_debug_group_dots(None, None, 1, 31, None, None) == C.E_INVAL
    f32 = lib.colibri_moe_layer_f32
    assert f32(ctypes.byref(cfg), None, 0, None, None, None, None, None, None, 0, None, None, 0, None) == C.OK
    assert f32(ctypes.byref(cfg), None, 33, None, None, None, None, None, None, 0, None, None, 0, None) == C.E_INVAL
    assert f32(ctypes.byref(cfg), None, 4, None, None, None, None, None, None, 0, None, None, 0, None) == C.E_INVAL
    # the host-buffer entry: T == 0 is a no-op; missing buffers, missing given ids and a
    # short workspace are refused before any copy (the workspace address is never used)
    host = lib.colibri_moe_layer_host
    x = np.zeros((4, synth.TINY.d), np.float32)
    out = np.zeros_like(x)
    fake_ws = 1 << 20
    assert host(ctypes.byref(cfg), None, 0, None, None, None, None, None, None, 0, None, None, 0, None) == C.OK
    assert host(ctypes.byref(cfg), None, 4, None, None, None, None, None, None, 0, out.ctypes.data,
                fake_ws, 1 << 40, None) == C.E_INVAL
    assert host(ctypes.byref(cfg), x.ctypes.data, 4, None, None, None, None, None, None, 1, out.ctypes.data,
                fake_ws, 1 << 40, None) == C.E_INVAL
    assert host(ctypes.byref(cfg), x.ctypes.data, 4, None, None, None, None, None, None, 0, out.ctypes.data,
                fake_ws + 16, 1 << 40, None) == C.E_INVAL
    need = C.colibri_moe_host_workspace_bytes(cfg, 4)
    assert host(ctypes.byref(cfg), x.ctypes.data, 4, None, None, None, None, None, None, 0, out.ctypes.data,
                fake_ws, need - 1, None) == C.E_NOMEM
    # the layer stack: sizes are decode only; n_layers, aliasing and the workspace size are
    # checked before anything is enqueued (fake addresses are never dereferenced)
    assert C.colibri_moe_stack_workspace_bytes(cfg, 32) > C.colibri_moe_workspace_bytes(cfg, 32)
    assert lib.colibri_moe_stack_workspace_bytes(ctypes.byref(cfg), 33) == 0
    stack = lib.colibri_moe_stack_decode
    fx, fo1, fo2 = 1 << 24, 1 << 25, 1 << 26
    lay = (C.StackLayer * 2)(C.StackLayer(None, fx, None, fx, None, fx, fx, fo1),
                             C.StackLayer(None, fx, None, fx, None, fx, fx, fo2))
    no_shared = C.layer_cfg(synth.TINY.replace(has_shared=False))
    ok_args = (fx, 4, 2, lay, 0, fake_ws)
    assert stack(ctypes.byref(no_shared), fx, 0, 2, lay, 0, None, 0, None) == C.OK           # T == 0
    assert stack(ctypes.byref(no_shared), fx, 4, 0, lay, 0, fake_ws, 1 << 40, None) == C.E_INVAL
    assert stack(ctypes.byref(no_shared), fx, 4, C.STACK_MAX + 1, lay, 0, fake_ws, 1 << 40, None) == C.E_INVAL
    assert stack(ctypes.byref(no_shared), fx, 33, 2, lay, 0, fake_ws, 1 << 40, None) == C.E_INVAL
    assert stack(ctypes.byref(cfg), *ok_args, 1 << 40, None) == C.E_INVAL                   # no shared expert
    alias = (C.StackLayer * 2)(C.StackLayer(None, fx, None, fx, None, fx, fx, fo1),
                               C.StackLayer(None, fx, None, fx, None, fx, fx, fo1))
    assert stack(ctypes.byref(no_shared), fx, 4, 2, alias, 0, fake_ws, 1 << 40, None) == C.E_INVAL
    own = (C.StackLayer * 2)(C.StackLayer(None, fx, None, fx, None, fx, fx, fo1),
                             C.StackLayer(fo2, fx, None, fx, None, fx, fx, fo2))    # writes its own input
    assert stack(ctypes.byref(no_shared), fx, 4, 2, own, 0, fake_ws, 1 << 40, None) == C.E_INVAL
    need = C.colibri_moe_stack_workspace_bytes(no_shared, 4)
    assert stack(ctypes.byref(no_shared), *ok_args, need - 1, None) == C.E_NOMEM
    assert lib.colibri_lru_trace(0, 0, None, None, None) == C.E_INVAL


def test_cache_prefetch_entry_points_check_arguments(lib):
    """The prefetch-queue entry points refuse a missing cache or bad counts before touching
    a device."""
    import ctypes as ct
    n = ct.c_int(7)
    assert lib.colibri_expert_cache_set_prefetch(None, None, 2, 1 << 20) == C.E_INVAL
    assert lib.colibri_expert_cache_wait(None, None, 100) == C.E_INVAL
    assert lib.colibri_expert_cache_pump(None, 4, ct.byref(n)) == C.E_INVAL


def test_cache_policy_matches_oracle(lib, orc):
    rng = np.random.default_rng(11)
    for cap in (1, 3, 8):
        kinds = rng.choice([0, 1, 1, 2, 2], size=4000).astype(np.int32)
        keys = rng.integers(0, 3 * cap + 2, 4000).astype(np.int64)
        assert np.array_equal(C.colibri_lru_trace(cap, kinds, keys), orc.lru_trace(cap, kinds, keys))


def test_cache_policy_thrash_and_reuse(lib):
    C_ = 16
    kinds = np.tile([0, 1], 20 * (C_ + 1)).astype(np.int32)
    keys = np.repeat(np.arange(20 * (C_ + 1)) % (C_ + 1), 2).astype(np.int64)
    assert C.colibri_lru_trace(C_, kinds, keys)[1::2].sum() == 0
    keys = np.repeat(np.arange(20 * C_) % C_, 2).astype(np.int64)
    kinds = np.tile([0, 1], 20 * C_).astype(np.int32)
    assert C.colibri_lru_trace(C_, kinds, keys)[1::2].sum() == 19 * C_


def test_cache_hot_policy_matches_oracle(lib, orc):
    rng = np.random.default_rng(12)
    for cap in (3, 8):
        for n_hot in (1, 2, cap // 2, cap):
            kinds = rng.choice([0, 1, 1, 1, 2], size=3000).astype(np.int32)
            # skewed keys, so that use counts differ and the hot set changes hands
            keys = np.minimum(rng.zipf(1.3, 3000), 4 * cap).astype(np.int64)
            assert np.array_equal(C.colibri_lru_trace_hot(cap, n_hot, kinds, keys),
                                  orc.lru_hot_trace(cap, n_hot, kinds, keys)), (cap, n_hot)
    assert lib.colibri_lru_trace_hot(2, 3, 0, None, None, None) == C.E_INVAL
