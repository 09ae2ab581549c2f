"""Seeded synthetic inputs for one routed MoE FFN layer.

This module only draws random tensors with the shapes and distributions of
the layer's workloads and lays expert weights out in the library's blob
format. It holds none of the layer's arithmetic (no quantiser, no router, no
matmul), so that the CUDA path and the CPU oracle can both take their inputs
from it without sharing any computation.

Workloads (synthetic, no checkpoint or dataset involved):
  * ``TINY``  -- d=512, ffn=256, 16 experts top-4, 4 groups keep 2, x2.5, one shared expert.
  * ``OLMOE`` -- d=2048, ffn=1024, 64 experts top-8, softmax router, no shared expert.
  * ``GLM52`` -- d=6144, ffn=2048, 256 experts top-8, 8 groups keep 4, x2.5, one shared
    expert of ffn=2048, Zipf-skewed router bias. Its int4 nibbles are 3*6144*2048/2 =
    18,874,368 bytes per expert, the "~19 MB" routed expert of the Colibri pages.

Distributions: activations N(0,1) (prefill rows additionally scaled by U(0.5, 2));
router weights N(0, 0.05); bias N(0, 0.01) (tiny) or b0 * r^-1.1 over a seeded
permutation of the experts (GLM-shaped); int4 codes uniform over [-8, 7] (uniform
random bytes, two offset-binary nibbles each); fp32 group scales |N(0, 0.02)|.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np

GROUP = 32
ALIGN = 256

# Stream tags keep the seeded streams of different tensors independent.
_TAG_EXPERT, _TAG_SHARED, _TAG_ROUTER, _TAG_X, _TAG_IDS = 11, 12, 13, 14, 15


@dataclass(frozen=True)
class LayerSpec:
    name: str
    d: int
    ffn: int
    n_exp: int
    top_k: int
    n_group: int = 1
    topk_group: int = 1
    router: str = "sigmoid"          # "sigmoid" (grouped, with bias) or "softmax"
    norm_topk: bool = True
    routed_scale: float = 1.0
    has_shared: bool = False
    shared_ffn: int = 0
    bias: str = "none"               # "none" | "normal" | "zipf"
    zipf_s: float = 1.1
    zipf_b0: float = 1.0
    group: int = 32                  # quantisation group: 32 or 64 elements per scale

    def replace(self, **kw) -> "LayerSpec":
        return dataclasses.replace(self, **kw)


TINY = LayerSpec("tiny", d=512, ffn=256, n_exp=16, top_k=4, n_group=4, topk_group=2,
                 router="sigmoid", norm_topk=True, routed_scale=2.5, has_shared=True,
                 shared_ffn=256, bias="normal")
OLMOE = LayerSpec("olmoe", d=2048, ffn=1024, n_exp=64, top_k=8, router="softmax",
                  norm_topk=False, routed_scale=1.0, has_shared=False, bias="none")
GLM52 = LayerSpec("glm52", d=6144, ffn=2048, n_exp=256, top_k=8, n_group=8, topk_group=4,
                  router="sigmoid", norm_topk=True, routed_scale=2.5, has_shared=True,
                  shared_ffn=2048, bias="zipf")

SPECS = {s.name: s for s in (TINY, OLMOE, GLM52)}

# The same layers with the 64-element groups of the pages' int4 containers.
TINY64 = TINY.replace(name="tiny_g64", group=64)
OLMOE64 = OLMOE.replace(name="olmoe_g64", group=64)
GLM52_64 = GLM52.replace(name="glm52_g64", group=64)
SPECS.update({s.name: s for s in (TINY64, OLMOE64, GLM52_64)})


@dataclass(frozen=True)
class BlobLayout:
    """Byte offsets of one expert inside its blob: w1 | w3 | w2 | s1 | s3 | s2.

    Logical tensors: w1, w3 [f][d/2] packed nibbles (gate, up); w2 [d][f/2] (down);
    s1, s3 [f][d/group] fp32; s2 [d][f/group] fp32. Each part starts on a 256-byte boundary
    and is stored in row blocks (see ``pack_nibbles`` / ``pack_scales``).
    """
    d: int
    f: int
    w1: int
    w3: int
    w2: int
    s1: int
    s3: int
    s2: int
    nbytes: int

    @property
    def nibble_bytes(self) -> int:
        return 3 * self.d * self.f // 2


def _up(n: int) -> int:
    return (n + ALIGN - 1) // ALIGN * ALIGN


def blob_layout(d: int, f: int, group: int = GROUP) -> BlobLayout:
    if group not in (32, 64) or d % group or f % group:
        raise ValueError("d and f must be multiples of the group (32 or 64)")
    sizes = [f * d // 2, f * d // 2, d * f // 2,
             4 * f * (d // group), 4 * f * (d // group), 4 * d * (f // group)]
    offs, o = [], 0
    for s in sizes:
        offs.append(o)
        o = _up(o + s)
    return BlobLayout(d, f, *offs, o)


# Storage order of one packed int4 matrix W [R][K] (R, K multiples of 32): row blocks of
# ROW_BLOCK rows; inside a block, group-major: the 16 bytes of group g (columns 32g..32g+31)
# of the block's 32 rows lie together, row after row. Byte (r, g, j) is at
#     ((r // 32) * (K // 32) + g) * 512 + (r % 32) * 16 + j,
# and byte j of a group holds column 32g+2j in its low nibble, 32g+2j+1 in its high nibble.
# Scales S [R][K/32] follow the same order: S[r][g] at ((r // 32) * (K // 32) + g) * 32 + r % 32.
# With 64-element groups the nibbles are stored the same way (a 64-group is two
# consecutive 32-column tiles) and the scales S [R][K/64] at ((r // 32) * (K // 64) + g) * 32
# + r % 32.
ROW_BLOCK = 32


def pack_nibbles(w: np.ndarray) -> np.ndarray:
    """Logical packed matrix [R][K/2] (uint8, row-major) -> stored bytes (flat)."""
    R, H = w.shape
    assert R % ROW_BLOCK == 0 and H % 16 == 0
    return np.ascontiguousarray(w.reshape(R // ROW_BLOCK, ROW_BLOCK, H // 16, 16).transpose(0, 2, 1, 3)).reshape(-1)


def unpack_nibbles(flat: np.ndarray, R: int, K: int) -> np.ndarray:
    """Stored bytes (flat) -> logical packed matrix [R][K/2]."""
    H = K // 2
    b = flat[:R * H].reshape(R // ROW_BLOCK, H // 16, ROW_BLOCK, 16)
    return np.ascontiguousarray(b.transpose(0, 2, 1, 3)).reshape(R, H)


def pack_scales(s: np.ndarray) -> np.ndarray:
    """Logical scales [R][K/group] (fp32) -> stored order (flat fp32)."""
    R, NG = s.shape
    assert R % ROW_BLOCK == 0
    return np.ascontiguousarray(s.reshape(R // ROW_BLOCK, ROW_BLOCK, NG).transpose(0, 2, 1)).reshape(-1)


def unpack_scales(flat: np.ndarray, R: int, K: int, group: int = GROUP) -> np.ndarray:
    """Stored scales (flat fp32) -> logical [R][K/group]."""
    NG = K // group
    b = flat[:R * NG].reshape(R // ROW_BLOCK, NG, ROW_BLOCK)
    return np.ascontiguousarray(b.transpose(0, 2, 1)).reshape(R, NG)


def _parts(d: int, f: int, group: int = GROUP):
    """(name, offset, rows R, columns K) of the six parts of a blob."""
    L = blob_layout(d, f, group)
    return L, (("w1", L.w1, f, d), ("w3", L.w3, f, d), ("w2", L.w2, d, f),
               ("s1", L.s1, f, d), ("s3", L.s3, f, d), ("s2", L.s2, d, f))


def expert_views(blob: np.ndarray, d: int, f: int, group: int = GROUP) -> dict:
    """The logical tensors of one expert blob (uint8, length blob_layout(d, f, group).nbytes):
    w1, w3 [f][d/2], w2 [d][f/2] uint8 and s1, s3 [f][d/group], s2 [d][f/group] fp32 (copies)."""
    L, parts = _parts(d, f, group)
    b = blob.reshape(-1)
    assert b.dtype == np.uint8 and b.size >= L.nbytes
    out = {}
    for name, off, R, K in parts:
        if name[0] == "w":
            out[name] = unpack_nibbles(b[off:off + R * K // 2], R, K)
        else:
            out[name] = unpack_scales(b[off:off + 4 * R * (K // group)].view(np.float32), R, K, group)
    return out


def write_expert(out: np.ndarray, d: int, f: int, tensors: dict, group: int = GROUP) -> np.ndarray:
    """Store logical tensors (the keys of ``expert_views``) into a blob."""
    L, parts = _parts(d, f, group)
    b = out.reshape(-1)
    b[:L.nbytes] = 0
    for name, off, R, K in parts:
        if name[0] == "w":
            b[off:off + R * K // 2] = pack_nibbles(np.asarray(tensors[name], np.uint8))
        else:
            b[off:off + 4 * R * (K // group)] = pack_scales(np.asarray(tensors[name], np.float32)).view(np.uint8)
    return out


def fill_expert_blob(out: np.ndarray, d: int, f: int, seed: int, layer: int, expert: int,
                     shared: bool = False, group: int = GROUP) -> np.ndarray:
    """Draw one expert (uniform int4 codes, |N(0, 0.02)| scales) into ``out`` (uint8 blob).
    Codes and scales are i.i.d., so they are drawn straight into storage order."""
    L, parts = _parts(d, f, group)
    rng = np.random.default_rng([seed, layer, expert, _TAG_SHARED if shared else _TAG_EXPERT])
    b = out.reshape(-1)
    b[:L.nbytes] = 0
    for name, off, R, K in parts:
        if name[0] == "w":
            n = R * K // 2
            b[off:off + n] = np.frombuffer(rng.bytes(n), np.uint8)
        else:
            n = R * (K // group)
            s = np.abs(rng.standard_normal(n, dtype=np.float32)) * np.float32(0.02)
            b[off:off + 4 * n] = s.view(np.uint8)
    return out


def expert_blob(spec: LayerSpec, seed: int, layer: int, expert: int, shared: bool = False) -> np.ndarray:
    f = spec.shared_ffn if shared else spec.ffn
    blob = np.empty(blob_layout(spec.d, f, spec.group).nbytes, np.uint8)
    return fill_expert_blob(blob, spec.d, f, seed, layer, expert, shared, spec.group)


def router_weights(spec: LayerSpec, seed: int, layer: int = 0):
    """(Wr [E, d] fp32 ~ N(0, 0.05), bias [E] fp32 or None)."""
    rng = np.random.default_rng([seed, layer, 0, _TAG_ROUTER])
    Wr = rng.standard_normal((spec.n_exp, spec.d), dtype=np.float32) * np.float32(0.05)
    if spec.bias == "none":
        bias = None
    elif spec.bias == "normal":
        bias = rng.standard_normal(spec.n_exp, dtype=np.float32) * np.float32(0.01)
    elif spec.bias == "zipf":
        perm = rng.permutation(spec.n_exp)
        ranks = np.arange(1, spec.n_exp + 1, dtype=np.float64)
        bias = np.empty(spec.n_exp, np.float32)
        bias[perm] = (spec.zipf_b0 * ranks ** (-spec.zipf_s)).astype(np.float32)
    else:
        raise ValueError(spec.bias)
    return Wr, bias


def activations(spec: LayerSpec, seed: int, T: int, step: int = 0, row_scale: bool = False) -> np.ndarray:
    """x [T, d] fp32 ~ N(0, 1); with ``row_scale`` each row is multiplied by U(0.5, 2)."""
    rng = np.random.default_rng([seed, step, T, _TAG_X])
    x = rng.standard_normal((T, spec.d), dtype=np.float32)
    if row_scale:
        x *= rng.uniform(0.5, 2.0, size=(T, 1)).astype(np.float32)
    return x


@dataclass
class Layer:
    """One synthetic layer held in host memory."""
    spec: LayerSpec
    seed: int
    Wr: np.ndarray
    bias: np.ndarray | None
    blobs: np.ndarray            # [E, blob_bytes] uint8
    shared_blob: np.ndarray | None

    def expert(self, e: int) -> dict:
        """Logical tensors of routed expert e (unpacked once, then kept)."""
        memo = self.__dict__.setdefault("_views", {})
        if e not in memo:
            memo[e] = expert_views(self.blobs[e], self.spec.d, self.spec.ffn, self.spec.group)
        return memo[e]

    def shared(self) -> dict | None:
        if self.shared_blob is None:
            return None
        memo = self.__dict__.setdefault("_views", {})
        if "shared" not in memo:
            memo["shared"] = expert_views(self.shared_blob, self.spec.d, self.spec.shared_ffn, self.spec.group)
        return memo["shared"]


def make_layer(spec: LayerSpec, seed: int, layer: int = 0, experts=None) -> Layer:
    """Draw a whole layer. ``experts`` limits which routed experts are drawn (others stay zero)."""
    Wr, bias = router_weights(spec, seed, layer)
    nb = blob_layout(spec.d, spec.ffn, spec.group).nbytes
    blobs = np.zeros((spec.n_exp, nb), np.uint8)
    for e in (range(spec.n_exp) if experts is None else experts):
        fill_expert_blob(blobs[e], spec.d, spec.ffn, seed, layer, e, group=spec.group)
    sh = expert_blob(spec, seed, layer, 0, shared=True) if spec.has_shared else None
    return Layer(spec, seed, Wr, bias, blobs, sh)


def zipf_weights(n: int, s: float) -> np.ndarray:
    r = np.arange(1, n + 1, dtype=np.float64)
    p = r ** (-s)
    return p / p.sum()


def streaming_ids(spec: LayerSpec, seed: int, n_layers: int, n_steps: int, reuse: float = 0.7):
    """Correlated decode routing for the expert-streaming workload.

    ids [n_steps, n_layers, k] int32 and weights [n_steps, n_layers, k] fp32. Each layer
    has its own seeded Zipf(s) popularity order over the experts. At step 0 every id is
    drawn from it; afterwards each of the k ids is kept from the previous step with
    probability ``reuse``, else redrawn from the layer's Zipf law, never repeating an id
    within the token. Weights are positive, sum to routed_scale per token.
    """
    rng = np.random.default_rng([seed, n_layers, n_steps, _TAG_IDS])
    E, k = spec.n_exp, spec.top_k
    p = zipf_weights(E, spec.zipf_s)
    perms = [rng.permutation(E) for _ in range(n_layers)]
    ids = np.empty((n_steps, n_layers, k), np.int32)
    for s in range(n_steps):
        for l in range(n_layers):
            cur: list[int] = []
            for i in range(k):
                if s > 0 and rng.random() < reuse and int(ids[s - 1, l, i]) not in cur:
                    cur.append(int(ids[s - 1, l, i]))
                    continue
                while True:
                    e = int(perms[l][rng.choice(E, p=p)])
                    if e not in cur:
                        break
                cur.append(e)
            ids[s, l] = cur
    u = rng.uniform(0.5, 1.5, size=(n_steps, n_layers, k))
    w = (u / u.sum(-1, keepdims=True) * spec.routed_scale).astype(np.float32)
    return ids, w
