"""Thin Python binding of libcolibri.so (the C ABI in include/colibri.h).

Argument marshalling only: every function takes torch tensors (device memory that
torch allocated) or numpy arrays (host memory), passes their addresses and sizes to
the C entry point of the same name, and raises ColibriError on a non-zero status.
All computation runs in the CUDA kernels of libcolibri.so. If the library is not
built, the first call raises: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcolibri.so")

OK, E_INVAL, E_CUDA, E_NOMEM, E_TIMEOUT, E_MISS, E_STAGE, E_DEVICE = 0, -1, -2, -3, -4, -5, -6, -7
GROUP = 32
ROUTER_SIGMOID_GROUPED, ROUTER_SOFTMAX = 0, 1


class ColibriError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} ({status})")
        self.status = status


class LayerCfg(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("ffn", ctypes.c_int), ("n_exp", ctypes.c_int),
                ("top_k", ctypes.c_int), ("n_group", ctypes.c_int), ("topk_group", ctypes.c_int),
                ("has_shared", ctypes.c_int), ("shared_ffn", ctypes.c_int), ("router", ctypes.c_int),
                ("norm_topk", ctypes.c_int), ("routed_scale", ctypes.c_float), ("group", ctypes.c_int)]


class Expert(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w1", "w3", "w2", "s1", "s3", "s2")]


class StackLayer(ctypes.Structure):
    """colibri_stack_layer: one layer's device pointers for colibri_moe_stack_decode
    (`shared` is a host pointer to an Expert)."""
    _fields_ = [("x", ctypes.c_void_p), ("Wr", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("experts", ctypes.c_void_p),
                ("shared", ctypes.c_void_p), ("ids", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("out", ctypes.c_void_p)]

STACK_MAX = 16


class BlobLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("w1", "w3", "w2", "s1", "s3", "s2", "nbytes")]


class WorkspaceView(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("qx", "sx", "offsets", "pairs", "hq", "hs", "y", "fmax",
                                               "hs_stride", "hbf")]


class CacheStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("lookups", "hits", "misses", "prefetch_staged",
                                              "prefetch_used", "prefetch_skipped", "evictions",
                                              "bytes_staged", "prefetch_throttled", "prefetch_cancelled",
                                              "prefetch_bytes")] + [("n_slots", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


_P, _I, _I64, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_PCFG = ctypes.POINTER(LayerCfg)

# name -> (restype, argtypes); every symbol include/colibri.h declares.
SIGNATURES = {
    "colibri_blob_layout_for": (_I, [_I, _I, ctypes.POINTER(BlobLayout)]),
    "colibri_blob_layout_for_g": (_I, [_I, _I, _I, ctypes.POINTER(BlobLayout)]),
    "colibri_strerror": (ctypes.c_char_p, [_I]),
    "colibri_q8_quantize": (_I, [_P, _I, _I, _P, _P, _P]),
    "colibri_q8_quantize_g": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "colibri_router_topk": (_I, [_PCFG, _P, _I, _P, _P, _P, _P, _P, _P]),
    "colibri_moe_workspace_bytes": (_SZ, [_PCFG, _I]),
    "colibri_moe_stack_workspace_bytes": (_SZ, [_PCFG, _I]),
    "colibri_moe_stack_decode": (_I, [_PCFG, _P, _I, _I, ctypes.POINTER(StackLayer), _I, _P, _SZ, _P]),
    "colibri_moe_layer": (_I, [_PCFG, _P, _I, _P, _P, _P, ctypes.POINTER(Expert), _P, _P, _I, _P, _P,
                               _SZ, _P]),
    "colibri_moe_f32_workspace_bytes": (_SZ, [_PCFG, _I]),
    "colibri_moe_layer_f32": (_I, [_PCFG, _P, _I, _P, _P, _P, ctypes.POINTER(Expert), _P, _P, _I, _P, _P,
                                   _SZ, _P]),
    "colibri_moe_host_workspace_bytes": (_SZ, [_PCFG, _I]),
    "colibri_moe_layer_host": (_I, [_PCFG, _P, _I, _P, _P, _P, ctypes.POINTER(Expert), _P, _P, _I, _P, _P,
                                    _SZ, _P]),
    "colibri_moe_layer_noalloc": (_I, [_PCFG, _P, _I, _P, _P, _P, ctypes.POINTER(Expert), _P, _P, _I,
                                       _P, _P]),
    "colibri_workspace_status": (_I, [_PCFG, _I, _P, ctypes.POINTER(_I), _P]),
    "colibri_moe_workspace_view": (_I, [_PCFG, _I, ctypes.POINTER(WorkspaceView)]),
    "colibri_debug_group_dots": (_I, [_P, _P, _I, _I, _P, _P]),
    "colibri_debug_umma_codes": (_I, [_P, _P, _I, _I, _P, _P]),
    "colibri_moe_profile_enable": (_I, [_I]),
    "colibri_moe_profile_read": (_I, [ctypes.POINTER(ctypes.c_float), _I]),
    "colibri_expert_cache_init": (_I, [ctypes.POINTER(_P), _P, _SZ, _P, _I, _I, _I, _I, _I, _P]),
    "colibri_expert_cache_stage": (_I, [_P, _I, _P, _I]),
    "colibri_expert_cache_lookup": (_I, [_P, _I, _P, _I, _P]),
    "colibri_expert_cache_table": (_P, [_P, _I]),
    "colibri_expert_cache_set_strict": (_I, [_P, _I]),
    "colibri_expert_cache_set_prefetch": (_I, [_P, _P, _I, ctypes.c_size_t]),
    "colibri_expert_cache_wait": (_I, [_P, _P, _I]),
    "colibri_expert_cache_pump": (_I, [_P, _I, _P]),
    "colibri_expert_cache_stats": (_I, [_P, ctypes.POINTER(CacheStats)]),
    "colibri_expert_cache_sync": (_I, [_P, _I]),
    "colibri_expert_cache_destroy": (None, [_P]),
    "colibri_expert_cache_inject_stage_failure": (_I, [_P, _I]),
    "colibri_lru_trace": (_I, [_I, _I64, _P, _P, _P]),
    "colibri_lru_trace_hot": (_I, [_I, _I, _I64, _P, _P, _P]),
    "colibri_expert_cache_set_hot": (_I, [_P, _I]),
}

_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libcolibri.so. Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"libcolibri.so is not built ({LIB_PATH}); run "
                                  "`python -m routed_expert_ffn_grouped_b300.build`")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
        return _lib


def strerror(status: int) -> str:
    return lib().colibri_strerror(status).decode()


def _check(fn: str, status: int):
    if status != OK:
        raise ColibriError(fn, status, strerror(status))


def _ptr(t) -> int | None:
    """Address of a torch tensor or numpy array; an int is taken as a raw address (the
    expert cache's device table); None stays None."""
    if t is None or isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def layer_cfg(spec) -> LayerCfg:
    """LayerCfg from a layer spec (any object with the synth.LayerSpec attributes)."""
    return LayerCfg(d=spec.d, ffn=spec.ffn, n_exp=spec.n_exp, top_k=spec.top_k,
                    n_group=spec.n_group, topk_group=spec.topk_group,
                    has_shared=int(spec.has_shared), shared_ffn=spec.shared_ffn,
                    router=ROUTER_SOFTMAX if spec.router == "softmax" else ROUTER_SIGMOID_GROUPED,
                    norm_topk=int(spec.norm_topk), routed_scale=spec.routed_scale,
                    group=getattr(spec, "group", GROUP))


def colibri_blob_layout_for(d: int, f: int, group: int = GROUP) -> BlobLayout:
    out = BlobLayout()
    if group == GROUP:
        _check("colibri_blob_layout_for", lib().colibri_blob_layout_for(d, f, ctypes.byref(out)))
    else:
        _check("colibri_blob_layout_for_g", lib().colibri_blob_layout_for_g(d, f, group, ctypes.byref(out)))
    return out


def colibri_q8_quantize(x, q, scale, stream=None, group: int = GROUP):
    rows, cols = x.shape
    if group == GROUP:
        _check("colibri_q8_quantize",
               lib().colibri_q8_quantize(_ptr(x), rows, cols, _ptr(q), _ptr(scale), _stream(stream)))
    else:
        _check("colibri_q8_quantize_g",
               lib().colibri_q8_quantize_g(_ptr(x), rows, cols, group, _ptr(q), _ptr(scale), _stream(stream)))


def colibri_router_topk(cfg: LayerCfg, x, Wr, bias, logits, ids, w, stream=None):
    T = x.shape[0]
    _check("colibri_router_topk",
           lib().colibri_router_topk(ctypes.byref(cfg), _ptr(x), T, _ptr(Wr), _ptr(bias), _ptr(logits),
                                     _ptr(ids), _ptr(w), _stream(stream)))


def colibri_moe_workspace_bytes(cfg: LayerCfg, T_max: int) -> int:
    n = lib().colibri_moe_workspace_bytes(ctypes.byref(cfg), T_max)
    if n == 0:
        raise ColibriError("colibri_moe_workspace_bytes", E_INVAL, "invalid configuration")
    return n


def colibri_moe_layer(cfg: LayerCfg, x, Wr, bias, experts, shared: Expert | None, ids, w, ids_given: bool,
                      out, workspace, stream=None):
    """experts: device tensor holding E colibri_expert structs (see DeviceLayer)."""
    T = x.shape[0]
    _check("colibri_moe_layer",
           lib().colibri_moe_layer(ctypes.byref(cfg), _ptr(x), T, _ptr(Wr), _ptr(bias), _ptr(experts),
                                   ctypes.byref(shared) if shared is not None else None, _ptr(ids), _ptr(w),
                                   int(bool(ids_given)), _ptr(out), _ptr(workspace), workspace.numel(),
                                   _stream(stream)))


def colibri_moe_stack_workspace_bytes(cfg: LayerCfg, T_max: int) -> int:
    n = lib().colibri_moe_stack_workspace_bytes(ctypes.byref(cfg), T_max)
    if n == 0:
        raise ColibriError("colibri_moe_stack_workspace_bytes", E_INVAL, "invalid configuration or T_max > 32")
    return n


def colibri_moe_stack_decode(cfg: LayerCfg, x, layers, ids_given: bool, workspace, stream=None):
    """Several decode layers in one launch. layers: per layer a dict with x (optional:
    the layer's own activations), Wr, bias, experts (device tensors or None), shared
    (Expert or None), ids, w, out (device tensors); a layer without x reads the previous
    layer's out (layer 0: x)."""
    T = x.shape[0]
    arr = (StackLayer * len(layers))()
    keep = []
    for i, y in enumerate(layers):
        sh = y.get("shared")
        if sh is not None:
            keep.append(sh)
        arr[i] = StackLayer(_ptr(y.get("x")), _ptr(y.get("Wr")), _ptr(y.get("bias")), _ptr(y["experts"]),
                            ctypes.addressof(sh) if sh is not None else None, _ptr(y["ids"]), _ptr(y["w"]),
                            _ptr(y["out"]))
    _check("colibri_moe_stack_decode",
           lib().colibri_moe_stack_decode(ctypes.byref(cfg), _ptr(x), T, len(layers), arr, int(bool(ids_given)),
                                          _ptr(workspace), workspace.numel(), _stream(stream)))


def colibri_moe_f32_workspace_bytes(cfg: LayerCfg, T_max: int) -> int:
    n = lib().colibri_moe_f32_workspace_bytes(ctypes.byref(cfg), T_max)
    if n == 0:
        raise ColibriError("colibri_moe_f32_workspace_bytes", E_INVAL, "invalid configuration or T_max > 32")
    return n


def colibri_moe_layer_f32(cfg: LayerCfg, x, Wr, bias, experts, shared: Expert | None, ids, w, ids_given: bool,
                          out, workspace, stream=None):
    """The layer on fp32 activations (decode, T <= 32); arguments as colibri_moe_layer."""
    T = x.shape[0]
    _check("colibri_moe_layer_f32",
           lib().colibri_moe_layer_f32(ctypes.byref(cfg), _ptr(x), T, _ptr(Wr), _ptr(bias), _ptr(experts),
                                       ctypes.byref(shared) if shared is not None else None, _ptr(ids), _ptr(w),
                                       int(bool(ids_given)), _ptr(out), _ptr(workspace), workspace.numel(),
                                       _stream(stream)))


def colibri_moe_host_workspace_bytes(cfg: LayerCfg, T_max: int) -> int:
    n = lib().colibri_moe_host_workspace_bytes(ctypes.byref(cfg), T_max)
    if n == 0:
        raise ColibriError("colibri_moe_host_workspace_bytes", E_INVAL, "invalid configuration")
    return n


def colibri_moe_layer_host(cfg: LayerCfg, x, Wr, bias, experts, shared: Expert | None, ids, w,
                           ids_given: bool, out, workspace, stream=None):
    """colibri_moe_layer on host buffers (numpy arrays or CPU tensors, pinned or not): x,
    out, and ids, w (inputs when ids_given, else optional outputs) live in host memory;
    Wr, bias, experts and workspace on the device. Returns when out holds the result."""
    T = x.shape[0]
    _check("colibri_moe_layer_host",
           lib().colibri_moe_layer_host(ctypes.byref(cfg), _ptr(x), T, _ptr(Wr), _ptr(bias), _ptr(experts),
                                        ctypes.byref(shared) if shared is not None else None, _ptr(ids),
                                        _ptr(w), int(bool(ids_given)), _ptr(out), _ptr(workspace),
                                        workspace.numel(), _stream(stream)))


NOALLOC_SCRATCH_BYTES = 16 << 20


def colibri_moe_layer_noalloc(cfg: LayerCfg, x, Wr, bias, experts, shared: Expert | None, ids, w,
                              ids_given: bool, out, stream=None):
    """colibri_moe_layer on the library's own fixed device scratch (no workspace argument)."""
    T = x.shape[0]
    _check("colibri_moe_layer_noalloc",
           lib().colibri_moe_layer_noalloc(ctypes.byref(cfg), _ptr(x), T, _ptr(Wr), _ptr(bias), _ptr(experts),
                                           ctypes.byref(shared) if shared is not None else None, _ptr(ids),
                                           _ptr(w), int(bool(ids_given)), _ptr(out), _stream(stream)))


def colibri_workspace_status(cfg: LayerCfg, T_max: int, workspace, stream=None) -> int:
    st = ctypes.c_int(0)
    _check("colibri_workspace_status",
           lib().colibri_workspace_status(ctypes.byref(cfg), T_max, _ptr(workspace), ctypes.byref(st),
                                          _stream(stream)))
    return st.value


def colibri_moe_workspace_view(cfg: LayerCfg, T_max: int) -> WorkspaceView:
    v = WorkspaceView()
    _check("colibri_moe_workspace_view", lib().colibri_moe_workspace_view(ctypes.byref(cfg), T_max, ctypes.byref(v)))
    return v


def colibri_debug_group_dots(w, qa, dots, rows: int, cols: int, stream=None):
    """w: a [rows][cols] packed int4 matrix in the stored layout (flat bytes)."""
    _check("colibri_debug_group_dots",
           lib().colibri_debug_group_dots(_ptr(w), _ptr(qa), rows, cols, _ptr(dots), _stream(stream)))


def colibri_debug_umma_codes(a, b, d, stream=None):
    """d[128][n] = a[128][k] . b[n][k]^T on the tensor core (int8 codes as bf16)."""
    n, k = b.shape
    _check("colibri_debug_umma_codes",
           lib().colibri_debug_umma_codes(_ptr(a), _ptr(b), n, k, _ptr(d), _stream(stream)))


PROFILE_KERNELS = ("q8", "router_logits", "router_select", "bucket", "gateup", "down", "combine")


def colibri_moe_profile_enable(on: bool):
    _check("colibri_moe_profile_enable", lib().colibri_moe_profile_enable(int(bool(on))))


def colibri_moe_profile_read() -> dict:
    ms = (ctypes.c_float * len(PROFILE_KERNELS))()
    _check("colibri_moe_profile_read", lib().colibri_moe_profile_read(ms, len(PROFILE_KERNELS)))
    return dict(zip(PROFILE_KERNELS, list(ms)))


def colibri_lru_trace(capacity: int, kinds, keys) -> np.ndarray:
    kinds = np.ascontiguousarray(kinds, np.int32)
    keys = np.ascontiguousarray(keys, np.int64)
    res = np.empty(len(kinds), np.int8)
    _check("colibri_lru_trace", lib().colibri_lru_trace(capacity, len(kinds), _ptr(kinds), _ptr(keys), _ptr(res)))
    return res


def colibri_lru_trace_hot(capacity: int, n_hot: int, kinds, keys) -> np.ndarray:
    kinds = np.ascontiguousarray(kinds, np.int32)
    keys = np.ascontiguousarray(keys, np.int64)
    res = np.empty(len(kinds), np.int8)
    _check("colibri_lru_trace_hot",
           lib().colibri_lru_trace_hot(capacity, n_hot, len(kinds), _ptr(kinds), _ptr(keys), _ptr(res)))
    return res


class ExpertCache:
    """colibri_expert_cache_* over a caller-owned HBM pool and pinned host blobs."""

    def __init__(self, pool, pinned_host, n_layers: int, n_exp: int, d: int, ffn: int, top_k: int,
                 copy_stream):
        self._pool, self._host, self._copy = pool, pinned_host, copy_stream
        h = ctypes.c_void_p()
        _check("colibri_expert_cache_init",
               lib().colibri_expert_cache_init(ctypes.byref(h), _ptr(pool), pool.numel() * pool.element_size(),
                                               _ptr(pinned_host), n_layers, n_exp, d, ffn, top_k,
                                               _stream(copy_stream)))
        self.handle = h

    def stage(self, layer: int, ids):
        ids = np.ascontiguousarray(ids, np.int32)
        _check("colibri_expert_cache_stage", lib().colibri_expert_cache_stage(self.handle, layer, _ptr(ids), ids.size))

    def lookup(self, layer: int, ids, wait_on=None):
        ids = np.ascontiguousarray(ids, np.int32)
        _check("colibri_expert_cache_lookup",
               lib().colibri_expert_cache_lookup(self.handle, layer, _ptr(ids), ids.size, _stream(wait_on)))

    def table(self, layer: int) -> int:
        p = lib().colibri_expert_cache_table(self.handle, layer)
        if not p:
            raise ColibriError("colibri_expert_cache_table", E_INVAL, "bad layer")
        return p

    def set_hot(self, n_hot: int):
        _check("colibri_expert_cache_set_hot", lib().colibri_expert_cache_set_hot(self.handle, int(n_hot)))

    def set_prefetch(self, prefetch_stream=None, max_in_flight: int = 0, chunk_bytes: int = 0):
        """Prefetches on their own stream (kept alive here): whole-blob copies, at most
        max_in_flight running (chunk_bytes 0), or queued chunks that wait() enqueues."""
        self._pcopy = prefetch_stream
        _check("colibri_expert_cache_set_prefetch",
               lib().colibri_expert_cache_set_prefetch(
                   self.handle, None if prefetch_stream is None else _stream(prefetch_stream), int(max_in_flight),
                   int(chunk_bytes)))

    def wait(self, stream=None, timeout_ms: int = 10000):
        """Waits for `stream`'s work so far, enqueuing queued prefetch chunks meanwhile."""
        _check("colibri_expert_cache_wait", lib().colibri_expert_cache_wait(self.handle, _stream(stream), timeout_ms))

    def pump(self, max_chunks: int) -> int:
        """Enqueues up to max_chunks queued prefetch chunks now; returns how many."""
        n = ctypes.c_int(0)
        _check("colibri_expert_cache_pump", lib().colibri_expert_cache_pump(self.handle, int(max_chunks),
                                                                             ctypes.byref(n)))
        return n.value

    def set_strict(self, strict: bool):
        _check("colibri_expert_cache_set_strict", lib().colibri_expert_cache_set_strict(self.handle, int(strict)))

    def stats(self) -> dict:
        st = CacheStats()
        _check("colibri_expert_cache_stats", lib().colibri_expert_cache_stats(self.handle, ctypes.byref(st)))
        return st.as_dict()

    def sync(self, timeout_ms: int = 10000):
        _check("colibri_expert_cache_sync", lib().colibri_expert_cache_sync(self.handle, timeout_ms))

    def inject_stage_failure(self, count: int):
        _check("colibri_expert_cache_inject_stage_failure",
               lib().colibri_expert_cache_inject_stage_failure(self.handle, count))

    def close(self):
        if self.handle:
            lib().colibri_expert_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DeviceLayer:
    """A synthetic layer uploaded to one GPU: expert blobs in one HBM tensor, the device
    table of E colibri_expert structs, the shared expert struct, Wr and bias."""

    def __init__(self, layer, device="cuda", experts=None):
        import torch
        spec = layer.spec
        self.spec = spec
        self.cfg = layer_cfg(spec)
        self.lay = colibri_blob_layout_for(spec.d, spec.ffn, getattr(spec, "group", GROUP))
        nb = self.lay.nbytes
        assert layer.blobs.shape[1] == nb
        self.blobs = torch.from_numpy(layer.blobs).to(device)
        self.Wr = torch.from_numpy(layer.Wr).to(device)
        self.bias = torch.from_numpy(layer.bias).to(device) if layer.bias is not None else None
        base = self.blobs.data_ptr()
        table = (Expert * spec.n_exp)()
        for e in range(spec.n_exp):
            table[e] = self._expert_at(base + e * nb, self.lay)
        self.table = torch.frombuffer(bytearray(bytes(table)), dtype=torch.uint8).to(device)
        self.shared = None
        self.shared_blob = None
        if spec.has_shared:
            self.shared_blob = torch.from_numpy(layer.shared_blob).to(device)
            sl = colibri_blob_layout_for(spec.d, spec.shared_ffn, getattr(spec, "group", GROUP))
            self.shared = self._expert_at(self.shared_blob.data_ptr(), sl)

    @classmethod
    def twin(cls, other: "DeviceLayer", shift: int = 1) -> "DeviceLayer":
        """Another layer of the same shape at other device addresses: the same expert blobs
        and shared expert copied on the device, router rows and bias rolled by `shift`
        experts (so the twin routes elsewhere). For runs that need a second layer without
        generating one on the host."""
        import torch
        t = cls.__new__(cls)
        t.spec, t.cfg, t.lay = other.spec, other.cfg, other.lay
        t.blobs = other.blobs.clone()
        t.Wr = torch.roll(other.Wr, shifts=shift, dims=0).contiguous()
        t.bias = torch.roll(other.bias, shifts=shift, dims=0).contiguous() if other.bias is not None else None
        base, nb = t.blobs.data_ptr(), t.lay.nbytes
        table = (Expert * t.spec.n_exp)()
        for e in range(t.spec.n_exp):
            table[e] = cls._expert_at(base + e * nb, t.lay)
        t.table = torch.frombuffer(bytearray(bytes(table)), dtype=torch.uint8).to(other.blobs.device)
        t.shared = None
        t.shared_blob = None
        if t.spec.has_shared:
            t.shared_blob = other.shared_blob.clone()
            sl = colibri_blob_layout_for(t.spec.d, t.spec.shared_ffn, getattr(t.spec, "group", GROUP))
            t.shared = cls._expert_at(t.shared_blob.data_ptr(), sl)
        return t

    @staticmethod
    def _expert_at(base: int, lay: BlobLayout) -> Expert:
        return Expert(base + lay.w1, base + lay.w3, base + lay.w2, base + lay.s1, base + lay.s3, base + lay.s2)
