"""CUDA path (through the C ABI) against the C oracle, on the same seeded inputs.

Bit-exact: q8 codes and scales, router logits, expert ids, int32 group dots, bucket
offsets and pair lists. Within tolerance: routing weights (1e-6 relative; fp64 sums in
another order) and layer outputs, max |out - oracle| <= 2e-3 * rms(oracle) in fp32.
"""
import numpy as np
import pytest

from routed_expert_ffn_grouped_b300 import synth

from h_codes import check_h_codes_and_output, h_codes_checked

pytestmark = pytest.mark.gpu

TOL = 2e-3


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


_layers = {}


def dev_layer(C, spec, seed=0):
    key = (spec, seed)
    if key not in _layers:
        host = synth.make_layer(spec, seed)
        _layers[key] = (host, C.DeviceLayer(host))
    return _layers[key]


def assert_rms_close(got, want, tol=TOL):
    want = np.asarray(want, np.float64)
    rms = np.sqrt(np.mean(want ** 2))
    err = np.max(np.abs(np.asarray(got, np.float64) - want)) if want.size else 0.0
    assert err <= tol * rms, f"max err {err:.3e} > {tol} * rms {rms:.3e}"


def to_dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# ------------------------------------------------------------------ q8
@pytest.mark.parametrize("rows,cols", [(1, 512), (4, 6144), (16, 2048), (2048, 6144), (3, 32)])
def test_q8_bit_exact(torch_cuda, C, orc, rows, cols):
    torch = torch_cuda
    rng = np.random.default_rng(rows * 7 + cols)
    x = (rng.standard_normal((rows, cols)) * rng.uniform(0.01, 50, (rows, 1))).astype(np.float32)
    x[0, :32] = 0.0                                   # an all-zero group
    g = 32 if cols >= 64 else 0
    x[-1, g:g + 32] = np.arange(32, dtype=np.float32) - 15.5   # exact half-points after scaling
    q = torch.empty((rows, cols), dtype=torch.int8, device="cuda")
    s = torch.empty((rows, cols // 32), dtype=torch.float32, device="cuda")
    C.colibri_q8_quantize(to_dev(torch, x), q, s)
    torch.cuda.synchronize()
    qo, so = orc.q8_quantize(x)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))


# ------------------------------------------------------------------ router
@pytest.mark.parametrize("name,T", [("tiny", 4), ("tiny", 37), ("olmoe", 1), ("olmoe", 16),
                                    ("glm52", 1), ("glm52", 4), ("glm52", 64)])
def test_router_bit_exact(torch_cuda, C, orc, name, T):
    torch = torch_cuda
    spec = synth.SPECS[name]
    Wr, bias = synth.router_weights(spec, 0)
    x = synth.activations(spec, 0, T, step=3)
    cfg = C.layer_cfg(spec)
    logits = torch.empty((T, spec.n_exp), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda")
    C.colibri_router_topk(cfg, to_dev(torch, x), to_dev(torch, Wr),
                          None if bias is None else to_dev(torch, bias), logits, ids, w)
    torch.cuda.synchronize()
    lo = orc.router_logits(x, Wr)
    assert np.array_equal(logits.cpu().numpy().view(np.uint32), lo.view(np.uint32))
    io, wo = orc.router_select(spec, lo, bias)
    assert np.array_equal(ids.cpu().numpy(), io)
    np.testing.assert_allclose(w.cpu().numpy(), wo, rtol=1e-6, atol=0)


def test_router_ties_lowest_index(torch_cuda, C, orc):
    """All-equal logits (x = 0): ids must be the lowest indices of the lowest groups."""
    torch = torch_cuda
    spec = synth.GLM52
    Wr, _ = synth.router_weights(spec, 0)
    x = np.zeros((2, spec.d), np.float32)
    cfg = C.layer_cfg(spec)
    logits = torch.empty((2, spec.n_exp), dtype=torch.float32, device="cuda")
    ids = torch.empty((2, spec.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((2, spec.top_k), dtype=torch.float32, device="cuda")
    C.colibri_router_topk(cfg, to_dev(torch, x), to_dev(torch, Wr), None, logits, ids, w)
    io, _ = orc.router_select(spec, orc.router_logits(x, Wr), None)
    assert np.array_equal(ids.cpu().numpy(), io)
    assert io[0].tolist() == list(range(8))


# ------------------------------------------------------------------ integer group dots
@pytest.mark.parametrize("rows,cols", [(64, 6144), (96, 2048), (32, 32)])
def test_group_dots_bit_exact(torch_cuda, C, orc, rows, cols):
    torch = torch_cuda
    rng = np.random.default_rng(rows + cols)
    w = rng.integers(0, 256, (rows, cols // 2), dtype=np.uint8)
    qa = rng.integers(-127, 128, cols).astype(np.int8)
    qa[:32] = -127
    w[0, :16] = 0                                       # -8 x -127 in group 0: 32512
    w[1, :16] = 0xFF                                    # 7 x -127 in group 0: -28448
    dots = torch.empty((rows, cols // 32), dtype=torch.int32, device="cuda")
    C.colibri_debug_group_dots(to_dev(torch, synth.pack_nibbles(w)), to_dev(torch, qa), dots,
                               rows=rows, cols=cols)
    torch.cuda.synchronize()
    want = orc.group_dots(w, qa)
    assert want[0, 0] == 32512 and want[1, 0] == -28448
    assert np.array_equal(dots.cpu().numpy(), want)


@pytest.mark.parametrize("n,k", [(16, 16), (16, 32), (64, 32), (128, 64), (256, 256)])
def test_umma_tile_integer_dots_exact(torch_cuda, C, n, k):
    """One tcgen05 tile of int4-range weight codes against int8 activation codes: the
    int32 result must equal the integer matmul exactly (brute force in int64)."""
    torch = torch_cuda
    rng = np.random.default_rng(n * 1000 + k)
    a = rng.integers(-8, 8, (128, k)).astype(np.int8)
    b = rng.integers(-127, 128, (n, k)).astype(np.int8)
    a[0, :32 if k >= 32 else k] = -8                  # the extreme group: -8 x -127 per element
    b[0, :32 if k >= 32 else k] = -127
    d = torch.empty((128, n), dtype=torch.int32, device="cuda")
    C.colibri_debug_umma_codes(to_dev(torch, a), to_dev(torch, b), d)
    torch.cuda.synchronize()
    want = a.astype(np.int64) @ b.astype(np.int64).T
    assert want[0, 0] == 1016 * min(k, 32) + (int(a[0, 32:].astype(np.int64) @ b[0, 32:].astype(np.int64)) if k > 32 else 0)
    assert np.array_equal(d.cpu().numpy().astype(np.int64), want)


# ------------------------------------------------------------------ the layer
def run_layer(torch, C, dl, x, ids=None, w=None):
    spec = dl.spec
    T = x.shape[0]
    cfg = dl.cfg
    ws = torch.empty(C.colibri_moe_workspace_bytes(cfg, max(T, 1)), dtype=torch.uint8, device="cuda")
    out = torch.empty((T, spec.d), dtype=torch.float32, device="cuda")
    given = ids is not None
    ids_d = to_dev(torch, ids) if given else torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
    w_d = to_dev(torch, w) if given else torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda")
    C.colibri_moe_layer(cfg, to_dev(torch, x), dl.Wr, dl.bias, dl.table, dl.shared, ids_d, w_d, given, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ids_d.cpu().numpy(), w_d.cpu().numpy(), ws


def ws_slice(ws, off, nbytes, dtype):
    return ws[off:off + nbytes].cpu().numpy().view(dtype)


def assert_buckets_exact(C, dl, ws, T, ids_o):
    """Bucket offsets and the pair list the layer left in its workspace: bit-exact against
    the oracle's stable counting sort of the oracle's ids (a non-stable scatter, or a wrong
    scan, fails here even where the outputs would agree)."""
    spec = dl.spec
    v = C.colibri_moe_workspace_view(dl.cfg, T)
    off = ws_slice(ws, v.offsets, 4 * (spec.n_exp + 1), np.int32)
    pairs = ws_slice(ws, v.pairs, 4 * T * spec.top_k, np.int32)
    off_o, pairs_o = orc_bucket(ids_o, spec.n_exp)
    assert np.array_equal(off, off_o), "bucket offsets differ"
    assert np.array_equal(pairs, pairs_o), "pair list differs"
    return off_o, pairs_o


def orc_bucket(ids, E):
    import oracle
    return oracle.bucket(ids, E)


@pytest.mark.parametrize("name,T", [("tiny", 4), ("tiny", 1), ("tiny", 13), ("olmoe", 1), ("olmoe", 16),
                                    ("glm52", 1), ("glm52", 4), ("glm52", 32)])
def test_moe_layer_parity(torch_cuda, C, orc, flip_report, name, T):
    torch = torch_cuda
    spec = synth.SPECS[name]
    host, dl = dev_layer(C, spec)
    x = synth.activations(spec, 0, T, step=11)
    out, ids, w, ws = run_layer(torch, C, dl, x)
    assert C.colibri_workspace_status(dl.cfg, T, ws) == C.OK
    ref, ids_o, w_o = orc.moe_layer(spec, x, host.Wr, host.bias, host.expert, host.shared())
    assert np.array_equal(ids, ids_o)
    np.testing.assert_allclose(w, w_o, rtol=1e-6)
    assert_rms_close(out, ref)
    if T * spec.top_k <= 64:
        # every pair's q8(h) codes and scales (larger batches: the sample below)
        n = check_h_codes_and_output(orc, C, spec, host, x, ids_o, w_o, ws, out, ref)
        flip_report(n, h_codes_checked(spec, T))
    # intermediates inside the workspace: q8 codes of x and the bucket lists, bit-exact
    v = C.colibri_moe_workspace_view(dl.cfg, T)
    qx = ws_slice(ws, v.qx, T * spec.d, np.int8).reshape(T, spec.d)
    sx = ws_slice(ws, v.sx, 4 * T * spec.d // 32, np.float32).reshape(T, -1)
    qo, so = orc.q8_quantize(x)
    assert np.array_equal(qx, qo) and np.array_equal(sx.view(np.uint32), so.view(np.uint32))
    off = ws_slice(ws, v.offsets, 4 * (spec.n_exp + 1), np.int32)
    pairs = ws_slice(ws, v.pairs, 4 * T * spec.top_k, np.int32)
    off_o, pairs_o = orc.bucket(ids_o, spec.n_exp)
    assert np.array_equal(off, off_o) and np.array_equal(pairs, pairs_o)
    # h codes: equal except a rounding-boundary flip of at most 1
    hq = ws_slice(ws, v.hq, (T * spec.top_k) * v.fmax, np.int8).reshape(-1, v.fmax)
    t, i = 0, 0
    _, qh_o, _ = orc.expert_token(host.expert(int(ids_o[t, i])), qo[t], so[t])
    diff = np.abs(hq[t * spec.top_k + i, :spec.ffn].astype(np.int32) - qh_o)
    assert diff.max() <= 1 and (diff == 0).mean() > 0.95


def test_moe_layer_ids_given(torch_cuda, C, orc):
    torch = torch_cuda
    spec = synth.GLM52
    host, dl = dev_layer(C, spec)
    ids, w = synth.streaming_ids(spec, 5, 1, 2)
    ids, w = ids[:, 0], w[:, 0]          # 2 tokens
    x = synth.activations(spec, 5, 2)
    out, ids_d, w_d, ws = run_layer(torch, C, dl, x, ids, w)
    assert np.array_equal(ids_d, ids)
    ref, _, _ = orc.moe_layer(spec, x, None, None, host.expert, host.shared(), ids=ids, w=w)
    assert_rms_close(out, ref)


def test_moe_layer_bad_id_reports(torch_cuda, C):
    torch = torch_cuda
    spec = synth.TINY
    _, dl = dev_layer(C, spec)
    ids = np.array([[0, 1, 2, spec.n_exp]], np.int32)         # last id out of range
    w = np.full((1, 4), 0.5, np.float32)
    _, _, _, ws = run_layer(torch, C, dl, synth.activations(spec, 0, 1), ids, w)
    assert C.colibri_workspace_status(dl.cfg, 1, ws) == C.E_DEVICE
    assert C.colibri_workspace_status(dl.cfg, 1, ws) == C.OK    # read clears it


@pytest.mark.parametrize("name,T,f32", [("tiny", 3, False), ("olmoe", 2, False), ("glm52", 1, False),
                                        ("glm52", 4, False), ("tiny", 40, False), ("glm52", 2, True)])
def test_router_nan_activation_ranks_lowest(torch_cuda, C, orc, name, T, f32):
    """A token with a NaN activation has NaN logits. Every selection (decode kernel,
    prefill and fp32-activation selection kernels) ranks a NaN score as -inf, so the layer
    still picks the oracle's ids (distinct and valid), reports no error and returns."""
    torch = torch_cuda
    spec = synth.SPECS[name]
    host, dl = dev_layer(C, spec)
    x = synth.activations(spec, 6, T)
    x[0, 5] = np.nan
    _, ids_d, _, ws = (run_layer_f32 if f32 else run_layer)(torch, C, dl, x)
    ids_o, _ = orc.router_topk(spec, x, host.Wr, host.bias)
    assert np.array_equal(ids_d, ids_o)
    assert C.colibri_workspace_status(dl.cfg, T, ws) == C.OK


def test_moe_layer_duplicate_id_reports(torch_cuda, C):
    """A token listing the same expert twice is bad input: the device flag reports it."""
    torch = torch_cuda
    spec = synth.TINY
    _, dl = dev_layer(C, spec)
    ids = np.array([[0, 1, 2, 3], [5, 6, 5, 7]], np.int32)
    w = np.full((2, 4), 0.5, np.float32)
    _, _, _, ws = run_layer(torch, C, dl, synth.activations(spec, 0, 2), ids, w)
    assert C.colibri_workspace_status(dl.cfg, 2, ws) == C.E_DEVICE


def test_moe_layer_empty_and_deterministic(torch_cuda, C):
    torch = torch_cuda
    spec = synth.OLMOE
    _, dl = dev_layer(C, spec)
    out, _, _, _ = run_layer(torch, C, dl, np.zeros((0, spec.d), np.float32))
    assert out.shape == (0, spec.d)
    x = synth.activations(spec, 1, 16)
    a, _, _, _ = run_layer(torch, C, dl, x)
    b, _, _, _ = run_layer(torch, C, dl, x)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("name,T", [("tiny", 33), ("tiny", 100), ("olmoe", 48)])
def test_prefill_gemm_parity(torch_cuda, C, orc, flip_report, name, T):
    """Batches above 32 tokens run the tcgen05 grouped GEMMs: every token against the
    oracle, ragged token tiles (counts not multiples of the 64-token tile) included; the
    prefill bucketing kernel's offsets and pair list bit-exact."""
    torch = torch_cuda
    spec = synth.SPECS[name]
    host, dl = dev_layer(C, spec)
    x = synth.activations(spec, 0, T, step=31, row_scale=True)
    out, ids, w, ws = run_layer(torch, C, dl, x)
    assert C.colibri_workspace_status(dl.cfg, T, ws) == C.OK
    ref, ids_o, w_o = orc.moe_layer(spec, x, host.Wr, host.bias, host.expert, host.shared())
    assert np.array_equal(ids, ids_o)
    np.testing.assert_allclose(w, w_o, rtol=1e-6)
    assert_rms_close(out, ref)
    assert_buckets_exact(C, dl, ws, T, ids_o)
    n = check_h_codes_and_output(orc, C, spec, host, x, ids_o, w_o, ws, out, ref)
    flip_report(n, h_codes_checked(spec, T))


def glm_prefill_check_tokens(counts, off_o, pairs_o, K, T, rng):
    """Tokens of the GLM-shaped T = 2048 batch whose outputs and q8(h) codes are compared
    with the oracle: the tokens of the last (ragged) 64-token tile and of the tile
    boundary of the three busiest experts, every token of four experts that fit one
    ragged tile (the fewest, a quarter, half and the most tokens below 64), and 64 more
    drawn at random."""
    picked = set()
    busiest = np.argsort(-counts, kind="stable")[:3]
    for e in busiest:
        b, c = int(off_o[e]), int(counts[e])
        last = ((c - 1) // 64) * 64
        for j in list(range(last, c)) + [j for j in (63, 64) if j < c]:
            picked.add(int(pairs_o[b + j]) // K)
    small = [int(e) for e in np.argsort(counts, kind="stable") if 0 < counts[e] < 64]
    if small:
        for q in (0, len(small) // 4, len(small) // 2, len(small) - 1):
            e = small[q]
            for j in range(int(counts[e])):
                picked.add(int(pairs_o[int(off_o[e]) + j]) // K)
    picked.update(int(t) for t in rng.choice(T, 64, replace=False))
    return sorted(picked)


def test_glm_prefill_t2048(torch_cuda, C, orc, flip_report):
    """The GLM-shaped prefill at its full size (T = 2048, Zipf-skewed expert loads):
    ids, weights, q8 codes of x and the bucket lists of all 16,384 pairs bit-exact or
    within 1e-6; outputs and every q8(h) code of a few hundred tokens chosen to cover the
    busiest experts' ragged and boundary tiles and whole lightly loaded experts (tokens
    are independent, so the oracle recomputes them alone)."""
    from concurrent.futures import ThreadPoolExecutor
    import os
    torch = torch_cuda
    spec = synth.GLM52
    host, dl = dev_layer(C, spec)
    T, K = 2048, spec.top_k
    x = synth.activations(spec, 0, T, step=21, row_scale=True)
    out, ids, w, ws = run_layer(torch, C, dl, x)
    assert C.colibri_workspace_status(dl.cfg, T, ws) == C.OK
    io_all, wo_all = orc.router_topk(spec, x, host.Wr, host.bias)
    assert np.array_equal(ids, io_all)
    np.testing.assert_allclose(w, wo_all, rtol=1e-6)
    v = C.colibri_moe_workspace_view(dl.cfg, T)
    qx = ws_slice(ws, v.qx, T * spec.d, np.int8).reshape(T, spec.d)
    sx = ws_slice(ws, v.sx, 4 * T * spec.d // 32, np.float32).reshape(T, -1)
    qo, so = orc.q8_quantize(x)
    assert np.array_equal(qx, qo) and np.array_equal(sx.view(np.uint32), so.view(np.uint32))
    off_o, pairs_o = assert_buckets_exact(C, dl, ws, T, io_all)
    counts = np.bincount(io_all.ravel(), minlength=spec.n_exp)
    assert counts.sum() == T * K and counts.max() > 64      # skewed: the busiest expert spans tiles
    toks = glm_prefill_check_tokens(counts, off_o, pairs_o, K, T, np.random.default_rng(7))
    assert len(toks) >= 100
    threads = max(1, min(16, os.cpu_count() or 1))
    chunks = [toks[i::threads] for i in range(threads) if toks[i::threads]]

    def ref_of(ch):
        r, _, _ = orc.moe_layer(spec, x[ch], host.Wr, host.bias, host.expert, host.shared())
        return ch, r

    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(ref_of, chunks))
    ref = np.empty((len(toks), spec.d), np.float32)
    pos = {t: j for j, t in enumerate(toks)}
    for ch, r in parts:
        for t, row in zip(ch, r):
            ref[pos[t]] = row
    n = check_h_codes_and_output(orc, C, spec, host, x, io_all, wo_all, ws, out[toks], ref,
                                 tokens=toks, threads=threads)
    flip_report(n, h_codes_checked(spec, len(toks)))


# d = 96: three 32-row blocks of d, so the down items' last pair has one block; ffn = 64:
# rows of q8(h) scales padded to 16 bytes; T * d not a multiple of 128: x staged by loads
ODD = synth.TINY.replace(name="odd96", d=96, ffn=64, n_exp=8, top_k=2, n_group=2, topk_group=1,
                         shared_ffn=64)


@pytest.mark.parametrize("T", [1, 3, 7])
def test_moe_layer_parity_odd_shape(torch_cuda, C, orc, flip_report, T):
    torch = torch_cuda
    host, dl = dev_layer(C, ODD)
    x = synth.activations(ODD, 0, T, step=3)
    out, ids, w, ws = run_layer(torch, C, dl, x)
    assert C.colibri_workspace_status(dl.cfg, T, ws) == C.OK
    ref, ids_o, w_o = orc.moe_layer(ODD, x, host.Wr, host.bias, host.expert, host.shared())
    assert np.array_equal(ids, ids_o)
    np.testing.assert_allclose(w, w_o, rtol=1e-6)
    assert_rms_close(out, ref)
    n = check_h_codes_and_output(orc, C, ODD, host, x, ids_o, w_o, ws, out, ref)
    flip_report(n, h_codes_checked(ODD, T))
    assert_buckets_exact(C, dl, ws, T, ids_o)




# The largest expert count and top_k the layer accepts (E = 1024 in 32 groups of 32,
# top_k = 32; up to 1,024 (token, expert) pairs at T = 32) on a small hidden size, and the
# degenerate routers: every expert picked, one expert per group, top-1 softmax. Decode
# runs the selection inside the expert kernel up to T x E = 4096 and in its own kernel
# above; T > 32 takes the grouped GEMMs.
MAXE = synth.TINY.replace(name="maxe1024", d=256, ffn=128, n_exp=1024, top_k=32, n_group=32, topk_group=4,
                          shared_ffn=128)
ALLK = synth.TINY.replace(name="allk8", n_exp=8, top_k=8, n_group=1, topk_group=1)
GS1 = synth.TINY.replace(name="gs1", n_exp=32, top_k=4, n_group=32, topk_group=8)
TOP1 = synth.TINY.replace(name="top1", n_exp=16, top_k=1, n_group=1, topk_group=1, router="softmax",
                          norm_topk=True, routed_scale=1.0, has_shared=False, shared_ffn=0, bias="none")


@pytest.mark.parametrize("spec,T", [(MAXE, 1), (MAXE, 4), (MAXE, 5), (MAXE, 32), (MAXE, 40),
                                    (ALLK, 1), (ALLK, 3), (ALLK, 40), (GS1, 1), (GS1, 2), (GS1, 33),
                                    (TOP1, 1), (TOP1, 7), (TOP1, 33)],
                         ids=lambda v: v.name if hasattr(v, "name") else str(v))
def test_moe_layer_parity_extreme_shapes(torch_cuda, C, orc, flip_report, spec, T):
    torch = torch_cuda
    host, dl = dev_layer(C, spec)
    x = synth.activations(spec, 0, T, step=5)
    out, ids, w, ws = run_layer(torch, C, dl, x)
    assert C.colibri_workspace_status(dl.cfg, T, ws) == C.OK
    ref, ids_o, w_o = orc.moe_layer(spec, x, host.Wr, host.bias, host.expert, host.shared())
    assert np.array_equal(ids, ids_o)
    np.testing.assert_allclose(w, w_o, rtol=1e-6)
    n = check_h_codes_and_output(orc, C, spec, host, x, ids_o, w_o, ws, out, ref)
    flip_report(n, h_codes_checked(spec, T))
    if spec is ALLK:
        assert all(sorted(r) == list(range(8)) for r in ids.tolist())
    if spec is TOP1:
        assert np.all(w == 1.0)
    # bucket lists in the workspace, bit-exact: the decode kernel's (T <= 32) and the
    # prefill bucketing kernel's (T > 32)
    assert_buckets_exact(C, dl, ws, T, ids_o)

# ------------------------------------------------------------------ host-buffer entry point
@pytest.mark.parametrize("name,T,pinned", [("glm52", 1, True), ("tiny", 13, False), ("olmoe", 16, True),
                                           ("tiny", 33, False)])
def test_moe_layer_host_entry(torch_cuda, C, orc, name, T, pinned):
    """colibri_moe_layer_host on host buffers: the same bits as colibri_moe_layer on device
    buffers (decode and prefill), so the same parity with the oracle."""
    torch = torch_cuda
    spec = synth.SPECS[name]
    host, dl = dev_layer(C, spec)
    x = synth.activations(spec, 0, T, step=13)
    out_dev, ids_dev, w_dev, _ = run_layer(torch, C, dl, x)
    ws = torch.empty(C.colibri_moe_host_workspace_bytes(dl.cfg, T), dtype=torch.uint8, device="cuda")
    if pinned:
        xh = torch.from_numpy(x).pin_memory()
        out = torch.empty((T, spec.d), dtype=torch.float32).pin_memory()
        ids = torch.empty((T, spec.top_k), dtype=torch.int32).pin_memory()
        w = torch.empty((T, spec.top_k), dtype=torch.float32).pin_memory()
    else:
        xh = np.ascontiguousarray(x)
        out = np.empty((T, spec.d), np.float32)
        ids = np.empty((T, spec.top_k), np.int32)
        w = np.empty((T, spec.top_k), np.float32)
    C.colibri_moe_layer_host(dl.cfg, xh, dl.Wr, dl.bias, dl.table, dl.shared, ids, w, False, out, ws)
    out, ids, w = (np.asarray(a) for a in (out, ids, w))
    assert np.array_equal(out.view(np.uint32), out_dev.view(np.uint32))
    assert np.array_equal(ids, ids_dev) and np.array_equal(w.view(np.uint32), w_dev.view(np.uint32))
    ref, ids_o, _ = orc.moe_layer(spec, x, host.Wr, host.bias, host.expert, host.shared())
    assert np.array_equal(ids, ids_o)
    assert_rms_close(out, ref)


def test_moe_layer_host_entry_repeated_pinned_calls(torch_cuda, C, orc):
    """Back-to-back calls on fresh page-locked buffers give the device entry's bits each
    time; a bad id reports the device status through the page-locked flag word, and the
    next good call is clean."""
    torch = torch_cuda
    spec = synth.TINY
    host, dl = dev_layer(C, spec)
    T = 3
    ws = torch.empty(C.colibri_moe_host_workspace_bytes(dl.cfg, T), dtype=torch.uint8, device="cuda")
    for step in range(4):
        x = synth.activations(spec, 1, T, step=50 + step)
        out_dev, ids_dev, w_dev, _ = run_layer(torch, C, dl, x)
        xh = torch.from_numpy(x).pin_memory()                   # a fresh buffer every call
        out = torch.empty((T, spec.d), dtype=torch.float32).pin_memory()
        ids = torch.empty((T, spec.top_k), dtype=torch.int32).pin_memory()
        w = torch.empty((T, spec.top_k), dtype=torch.float32).pin_memory()
        C.colibri_moe_layer_host(dl.cfg, xh, dl.Wr, dl.bias, dl.table, dl.shared, ids, w, False, out, ws)
        assert np.array_equal(out.numpy().view(np.uint32), out_dev.view(np.uint32)), step
        assert np.array_equal(ids.numpy(), ids_dev) and np.array_equal(w.numpy().view(np.uint32), w_dev.view(np.uint32))
    # ids given, pinned, one id out of range: the status comes back through the graph
    gid = torch.from_numpy(np.array([[0, 1, 2, 3], [4, 5, 6, 7], [8, 9, 10, spec.n_exp]], np.int32)).pin_memory()
    gw = torch.full((T, spec.top_k), 0.25, dtype=torch.float32).pin_memory()
    xh = torch.from_numpy(synth.activations(spec, 2, T)).pin_memory()
    out = torch.empty((T, spec.d), dtype=torch.float32).pin_memory()
    with pytest.raises(C.ColibriError) as e:
        C.colibri_moe_layer_host(dl.cfg, xh, None, None, dl.table, dl.shared, gid, gw, True, out, ws)
    assert e.value.status == C.E_DEVICE
    gid[2, 3] = 11
    C.colibri_moe_layer_host(dl.cfg, xh, None, None, dl.table, dl.shared, gid, gw, True, out, ws)
    ref, _, _ = orc.moe_layer(spec, xh.numpy(), None, None, host.expert, host.shared(), ids=gid.numpy(), w=gw.numpy())
    assert_rms_close(out.numpy(), ref)


def test_moe_layer_host_entry_ids_given_and_errors(torch_cuda, C, orc):
    torch = torch_cuda
    spec = synth.TINY
    host, dl = dev_layer(C, spec)
    ids = np.array([[0, 1, 2, 3], [5, 6, 4, 7]], np.int32)
    w = np.full((2, 4), 0.25, np.float32)
    x = synth.activations(spec, 2, 2)
    ws = torch.empty(C.colibri_moe_host_workspace_bytes(dl.cfg, 2), dtype=torch.uint8, device="cuda")
    out = np.empty((2, spec.d), np.float32)
    C.colibri_moe_layer_host(dl.cfg, x, None, None, dl.table, dl.shared, ids, w, True, out, ws)
    ref, _, _ = orc.moe_layer(spec, x, None, None, host.expert, host.shared(), ids=ids, w=w)
    assert_rms_close(out, ref)
    # an id out of range: the kernels skip it and the call returns the device status
    bad = ids.copy()
    bad[1, 2] = spec.n_exp
    with pytest.raises(C.ColibriError) as e:
        C.colibri_moe_layer_host(dl.cfg, x, None, None, dl.table, dl.shared, bad, w, True, out, ws)
    assert e.value.status == C.E_DEVICE
    # the next good call starts clean
    C.colibri_moe_layer_host(dl.cfg, x, None, None, dl.table, dl.shared, ids, w, True, out, ws)
    assert_rms_close(out, ref)
    # a workspace sized for the device entry alone is too short
    short = torch.empty(C.colibri_moe_workspace_bytes(dl.cfg, 2), dtype=torch.uint8, device="cuda")
    with pytest.raises(C.ColibriError) as e:
        C.colibri_moe_layer_host(dl.cfg, x, None, None, dl.table, dl.shared, ids, w, True, out, short)
    assert e.value.status == C.E_NOMEM


# ------------------------------------------------------------------ fp32-activation decode
def run_layer_f32(torch, C, dl, x, ids=None, w=None):
    spec = dl.spec
    T = x.shape[0]
    ws = torch.empty(C.colibri_moe_f32_workspace_bytes(dl.cfg, max(T, 1)), dtype=torch.uint8, device="cuda")
    out = torch.empty((T, spec.d), dtype=torch.float32, device="cuda")
    given = ids is not None
    ids_d = to_dev(torch, ids) if given else torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
    w_d = to_dev(torch, w) if given else torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda")
    C.colibri_moe_layer_f32(dl.cfg, to_dev(torch, x), dl.Wr, dl.bias, dl.table, dl.shared, ids_d, w_d, given,
                            out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ids_d.cpu().numpy(), w_d.cpu().numpy(), ws


@pytest.mark.parametrize("name,T", [("tiny", 1), ("tiny", 13), ("olmoe", 1), ("olmoe", 16), ("glm52", 1),
                                    ("glm52", 4), ("odd96", 3)])
def test_moe_layer_f32_parity(torch_cuda, C, orc, name, T):
    """Decode on fp32 activations against the oracle's fp32-activation layer: the same
    routing bit for bit, outputs within the layer's tolerance (nothing is quantised but
    the weights, so no code can round either way)."""
    torch = torch_cuda
    spec = ODD if name == "odd96" else synth.SPECS[name]
    host, dl = dev_layer(C, spec)
    x = synth.activations(spec, 0, T, step=17)
    out, ids, w, ws = run_layer_f32(torch, C, dl, x)
    assert C.colibri_workspace_status(dl.cfg, T, ws) == C.OK
    ref, ids_o, w_o = orc.moe_layer(spec, x, host.Wr, host.bias, host.expert, host.shared(), act="f32")
    assert np.array_equal(ids, ids_o)
    np.testing.assert_allclose(w, w_o, rtol=1e-6)
    assert_rms_close(out, ref)


def test_moe_layer_f32_ids_given_and_bad_id(torch_cuda, C, orc):
    torch = torch_cuda
    spec = synth.TINY
    host, dl = dev_layer(C, spec)
    ids = np.array([[0, 1, 2, 3], [5, 6, 5, 7]], np.int32)   # a repeated id is computed twice
    w = np.full((2, 4), 0.25, np.float32)
    x = synth.activations(spec, 4, 2)
    out, _, _, ws = run_layer_f32(torch, C, dl, x, ids, w)
    assert C.colibri_workspace_status(dl.cfg, 2, ws) == C.OK
    ref, _, _ = orc.moe_layer(spec, x, None, None, host.expert, host.shared(), ids=ids, w=w, act="f32")
    assert_rms_close(out, ref)
    bad = ids.copy()
    bad[0, 1] = spec.n_exp
    _, _, _, ws = run_layer_f32(torch, C, dl, x, bad, w)
    assert C.colibri_workspace_status(dl.cfg, 2, ws) == C.E_DEVICE
