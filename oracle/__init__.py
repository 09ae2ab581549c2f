"""Python front of the plain C oracle for one routed MoE FFN layer.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package. The CUDA library under
``routed_expert_ffn_grouped_b300`` never imports, links or calls it, and this
package imports nothing from there: the two share only the seeded inputs.

Every function takes and returns numpy arrays and calls the C oracle in
``colibri_oracle.c`` (built here with gcc). The C file states, per step, what
the method computes and which page passage it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "colibri_oracle.c")
_HDR = os.path.join(_HERE, "colibri_oracle.h")
_BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD_DIR, "libcolibri_oracle.so")

# Single-rounding fp32: no contraction into fma, no fast-math reassociation.
CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra"]

_lock = threading.Lock()
_lib = None

ROUTER_SIGMOID_GROUPED = 0
ROUTER_SOFTMAX = 1


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libcolibri_oracle.so`` (gcc)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= newest_src:
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


class Cfg(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("ffn", ctypes.c_int), ("n_exp", ctypes.c_int),
                ("top_k", ctypes.c_int), ("n_group", ctypes.c_int), ("topk_group", ctypes.c_int),
                ("has_shared", ctypes.c_int), ("shared_ffn", ctypes.c_int),
                ("router", ctypes.c_int), ("norm_topk", ctypes.c_int),
                ("routed_scale", ctypes.c_float)]


class Expert(ctypes.Structure):
    _fields_ = [("w1", ctypes.c_void_p), ("w3", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("s1", ctypes.c_void_p), ("s3", ctypes.c_void_p), ("s2", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(LIB_PATH)
            sig = {
                "orc_unpack_int4": (None, [_P, _I64, _P]),
                "orc_q8_quantize": (_I, [_P, _I64, _I64, _P, _P]),
                "orc_router_logits": (None, [_P, _I64, _I64, _P, _I64, _P]),
                "orc_router_select": (_I, [ctypes.POINTER(Cfg), _P, _I64, _P, _P, _P]),
                "orc_router_topk": (_I, [ctypes.POINTER(Cfg), _P, _I64, _P, _P, _P, _P]),
                "orc_bucket": (_I, [_P, _I64, _I, _I, _P, _P]),
                "orc_group_dots": (None, [_P, _P, _I64, _I64, _P]),
                "orc_expert_token": (_I, [_I, _I, ctypes.POINTER(Expert), _P, _P, _P, _P, _P, _P]),
                "orc_moe_layer": (_I, [ctypes.POINTER(Cfg), _P, _I64, _P, _P,
                                       ctypes.POINTER(Expert), ctypes.POINTER(Expert),
                                       _P, _P, _P, _P, _P]),
                "orc_expert_token_f32": (_I, [_I, _I, ctypes.POINTER(Expert), _P, _P, _P]),
                "orc_q8_quantize_g": (_I, [_P, _I64, _I64, _I, _P, _P]),
                "orc_group_dots_g": (_I, [_P, _P, _I64, _I64, _I, _P]),
                "orc_expert_token_g": (_I, [_I, _I, _I, ctypes.POINTER(Expert), _P, _P, _P, _P, _P, _P]),
                "orc_expert_token_f32_g": (_I, [_I, _I, _I, ctypes.POINTER(Expert), _P, _P, _P]),
                "orc_moe_layer_g": (_I, [ctypes.POINTER(Cfg), _I, _I, _P, _I64, _P, _P,
                                         ctypes.POINTER(Expert), ctypes.POINTER(Expert),
                                         _P, _P, _P, _P, _P]),
                "orc_moe_layer_f32": (_I, [ctypes.POINTER(Cfg), _P, _I64, _P, _P,
                                           ctypes.POINTER(Expert), ctypes.POINTER(Expert),
                                           _P, _P, _P, _P, _P]),
                "orc_lru_trace": (_I, [_I, _I64, _P, _P, _P]),
                "orc_lru_hot_trace": (_I, [_I, _I, _I64, _P, _P, _P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
        return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def make_cfg(spec) -> Cfg:
    """Oracle config from a layer spec (any object with the LayerSpec attributes)."""
    return Cfg(d=spec.d, ffn=spec.ffn, n_exp=spec.n_exp, top_k=spec.top_k,
               n_group=spec.n_group, topk_group=spec.topk_group,
               has_shared=int(spec.has_shared), shared_ffn=spec.shared_ffn,
               router=ROUTER_SOFTMAX if spec.router == "softmax" else ROUTER_SIGMOID_GROUPED,
               norm_topk=int(spec.norm_topk), routed_scale=spec.routed_scale)


def make_expert(views: dict) -> tuple[Expert, list]:
    """Expert struct over a dict of numpy arrays w1, w3, w2, s1, s3, s2 (kept alive by the list)."""
    keep = [_c(views[k], np.uint8 if k[0] == "w" else np.float32)
            for k in ("w1", "w3", "w2", "s1", "s3", "s2")]
    ex = Expert(*[a.ctypes.data for a in keep])
    return ex, keep


def unpack_int4(packed: np.ndarray) -> np.ndarray:
    p = _c(packed, np.uint8)
    q = np.empty(p.shape[:-1] + (2 * p.shape[-1],), np.int8)
    lib().orc_unpack_int4(_ptr(p), p.size, _ptr(q))
    return q


def q8_quantize(x: np.ndarray, group: int = 32):
    """q8 codes and scales per `group` (32 or 64) elements of each row."""
    x = _c(x, np.float32)
    rows, cols = (1, x.shape[0]) if x.ndim == 1 else x.shape
    q = np.empty(x.shape, np.int8)
    s = np.empty(x.shape[:-1] + (cols // group,), np.float32)
    if group == 32:
        rc = lib().orc_q8_quantize(_ptr(x), rows, cols, _ptr(q), _ptr(s))
    else:
        rc = lib().orc_q8_quantize_g(_ptr(x), rows, cols, group, _ptr(q), _ptr(s))
    if rc:
        raise ValueError("orc_q8_quantize: bad sizes")
    return q, s


def router_logits(x: np.ndarray, Wr: np.ndarray) -> np.ndarray:
    x, Wr = _c(x, np.float32), _c(Wr, np.float32)
    T, d = x.shape
    E = Wr.shape[0]
    out = np.empty((T, E), np.float32)
    lib().orc_router_logits(_ptr(x), T, d, _ptr(Wr), E, _ptr(out))
    return out


def router_select(spec_or_cfg, logits: np.ndarray, bias):
    cfg = spec_or_cfg if isinstance(spec_or_cfg, Cfg) else make_cfg(spec_or_cfg)
    logits = _c(logits, np.float32)
    T = logits.shape[0]
    ids = np.empty((T, cfg.top_k), np.int32)
    w = np.empty((T, cfg.top_k), np.float32)
    b = None if bias is None else _c(bias, np.float32)
    rc = lib().orc_router_select(ctypes.byref(cfg), _ptr(logits), T, _ptr(b), _ptr(ids), _ptr(w))
    if rc:
        raise ValueError("orc_router_select: bad config")
    return ids, w


def router_topk(spec_or_cfg, x, Wr, bias):
    cfg = spec_or_cfg if isinstance(spec_or_cfg, Cfg) else make_cfg(spec_or_cfg)
    x, Wr = _c(x, np.float32), _c(Wr, np.float32)
    T = x.shape[0]
    ids = np.empty((T, cfg.top_k), np.int32)
    w = np.empty((T, cfg.top_k), np.float32)
    b = None if bias is None else _c(bias, np.float32)
    rc = lib().orc_router_topk(ctypes.byref(cfg), _ptr(x), T, _ptr(Wr), _ptr(b), _ptr(ids), _ptr(w))
    if rc:
        raise ValueError("orc_router_topk: bad config")
    return ids, w


def bucket(ids: np.ndarray, E: int):
    ids = _c(ids, np.int32)
    T, k = ids.shape
    offsets = np.empty(E + 1, np.int32)
    pairs = np.empty(T * k, np.int32)
    rc = lib().orc_bucket(_ptr(ids), T, k, E, _ptr(offsets), _ptr(pairs))
    if rc:
        raise ValueError("orc_bucket: id out of range")
    return offsets, pairs


def group_dots(w_packed: np.ndarray, qa: np.ndarray, group: int = 32) -> np.ndarray:
    w, qa = _c(w_packed, np.uint8), _c(qa, np.int8)
    rows, cols = w.shape[0], 2 * w.shape[1]
    if group not in (32, 64) or cols % group:
        raise ValueError("group_dots: bad group")
    out = np.empty((rows, cols // group), np.int32)
    if group == 32:
        lib().orc_group_dots(_ptr(w), _ptr(qa), rows, cols, _ptr(out))
    elif lib().orc_group_dots_g(_ptr(w), _ptr(qa), rows, cols, group, _ptr(out)) != 0:
        raise ValueError("group_dots: the oracle rejected the group size")
    return out


def expert_token(views: dict, qx: np.ndarray, sx: np.ndarray, want_h: bool = False, group: int = 32):
    """One token through one expert; returns (y, qh, sh), and the fp32 h that (qh, sh)
    quantise as a fourth item when want_h. group: the quantisation group (32 or 64) of the
    expert's scales and of the activations."""
    ex, keep = make_expert(views)
    f = keep[0].shape[0]
    d = 2 * keep[0].shape[1]
    qx, sx = _c(qx, np.int8), _c(sx, np.float32)
    y = np.empty(d, np.float32)
    qh = np.empty(f, np.int8)
    sh = np.empty(f // group, np.float32)
    h = np.empty(f, np.float32) if want_h else None
    if group == 32:
        rc = lib().orc_expert_token(d, f, ctypes.byref(ex), _ptr(qx), _ptr(sx), _ptr(y), _ptr(qh), _ptr(sh),
                                    _ptr(h) if want_h else None)
    else:
        rc = lib().orc_expert_token_g(d, f, group, ctypes.byref(ex), _ptr(qx), _ptr(sx), _ptr(y), _ptr(qh),
                                      _ptr(sh), _ptr(h) if want_h else None)
    if rc:
        raise MemoryError("orc_expert_token")
    return (y, qh, sh, h) if want_h else (y, qh, sh)


def expert_token_f32(views: dict, x: np.ndarray, group: int = 32):
    """One token through one expert on fp32 activations; returns (y, h)."""
    ex, keep = make_expert(views)
    f = keep[0].shape[0]
    d = 2 * keep[0].shape[1]
    x = _c(x, np.float32)
    y = np.empty(d, np.float32)
    h = np.empty(f, np.float32)
    if group == 32:
        rc = lib().orc_expert_token_f32(d, f, ctypes.byref(ex), _ptr(x), _ptr(y), _ptr(h))
    else:
        rc = lib().orc_expert_token_f32_g(d, f, group, ctypes.byref(ex), _ptr(x), _ptr(y), _ptr(h))
    if rc:
        raise ValueError("orc_expert_token_f32: bad sizes")
    return y, h


def moe_layer(spec_or_cfg, x, Wr, bias, experts, shared=None, ids=None, w=None, act="q8", group=32):
    """The whole layer; ``experts`` is a list of E view dicts (or a callable e -> view dict,
    used only for the selected ids). act = "q8" (int8 activations, the layer's main form)
    or "f32" (fp32 activations); group = 32 or 64 (the quantisation group of the experts'
    scales and of the activations). Returns (out, ids, w)."""
    if act not in ("q8", "f32") or group not in (32, 64):
        raise ValueError((act, group))
    cfg = spec_or_cfg if isinstance(spec_or_cfg, Cfg) else make_cfg(spec_or_cfg)
    x = _c(x, np.float32)
    T = x.shape[0]
    E = cfg.n_exp
    if ids is None:
        ids_r, w_r = router_topk(cfg, x, Wr, bias) if T else (np.empty((0, cfg.top_k), np.int32),
                                                               np.empty((0, cfg.top_k), np.float32))
    else:
        ids_r, w_r = _c(ids, np.int32), _c(w, np.float32)
    table = (Expert * E)()
    keep = []
    needed = set(int(e) for e in ids_r.ravel())
    for e in range(E):
        if callable(experts):
            if e not in needed:
                continue
            v = experts(e)
        else:
            v = experts[e]
        ex, k = make_expert(v)
        table[e] = ex
        keep.append(k)
    sh_ex = None
    if cfg.has_shared:
        sh_ex, k = make_expert(shared)
        keep.append(k)
    out = np.empty((T, cfg.d), np.float32)
    if group == 32:
        fn = lib().orc_moe_layer if act == "q8" else lib().orc_moe_layer_f32
    else:
        def fn(cfg_p, *rest):
            return lib().orc_moe_layer_g(cfg_p, group, int(act == "f32"), *rest)
    rc = fn(ctypes.byref(cfg), _ptr(x), T, None if Wr is None else _ptr(_c(Wr, np.float32)),
                             None if bias is None else _ptr(_c(bias, np.float32)), table,
                             ctypes.byref(sh_ex) if sh_ex is not None else None,
                             _ptr(ids_r), _ptr(w_r), None, None, _ptr(out))
    if rc:
        raise ValueError("orc_moe_layer: bad input")
    return out, ids_r, w_r


def lru_hot_trace(capacity: int, n_hot: int, kinds, keys) -> np.ndarray:
    """The cache policy with n_hot usage-pinned slots (results as lru_trace)."""
    kinds = _c(kinds, np.int32)
    keys = _c(keys, np.int64)
    res = np.empty(len(kinds), np.int8)
    rc = lib().orc_lru_hot_trace(capacity, n_hot, len(kinds), _ptr(kinds), _ptr(keys), _ptr(res))
    if rc:
        raise ValueError("orc_lru_hot_trace: bad capacity or n_hot")
    return res


def lru_trace(capacity: int, kinds, keys) -> np.ndarray:
    kinds = _c(kinds, np.int32)
    keys = _c(keys, np.int64)
    res = np.empty(len(kinds), np.int8)
    rc = lib().orc_lru_trace(capacity, len(kinds), _ptr(kinds), _ptr(keys), _ptr(res))
    if rc:
        raise ValueError("orc_lru_trace: bad capacity")
    return res
