"""Several decode layers in one launch (colibri_moe_stack_decode) against the same layers
called one after another (colibri_moe_layer, each call's x the previous call's out), bit
for bit: every layer's output, ids and weights. Also the stack's own argument checks and
its device error path (a bad given id stops every layer, reported through the flag)."""
import numpy as np
import pytest

from routed_expert_ffn_grouped_b300 import synth

pytestmark = pytest.mark.gpu


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


_stacks = {}


def stack_layers(C, name, L):
    """L device layers of one shape: drawn layer by layer for the small shapes, else one
    drawn layer and twins of it with router rows rolled (each routes differently)."""
    key = (name, L)
    if key not in _stacks:
        spec = synth.SPECS[name]
        if spec.n_exp * spec.d * spec.ffn <= 64 * 2048 * 1024:  # tiny and OLMoE shapes
            layers = [C.DeviceLayer(synth.make_layer(spec, 0, layer=l)) for l in range(L)]
        else:
            base = C.DeviceLayer(synth.make_layer(spec, 0))
            layers = [base] + [C.DeviceLayer.twin(base, shift=7 * l) for l in range(1, L)]
        _stacks[key] = layers
    return _stacks[key]


def given_routing(spec, T, L, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([np.stack([rng.choice(spec.n_exp, spec.top_k, replace=False) for _ in range(T)])
                    for _ in range(L)]).astype(np.int32)
    w = rng.uniform(0.05, 1.0, (L, T, spec.top_k)).astype(np.float32)
    return ids, w


def run_sequential(torch, C, layers, x, ids_given, gids, gw, xs=None):
    """xs: per-layer activations (None: chained, layer l reads layer l - 1's out)."""
    spec, cfg = layers[0].spec, layers[0].cfg
    T = x.shape[0]
    ws = torch.empty(C.colibri_moe_workspace_bytes(cfg, T), dtype=torch.uint8, device="cuda")
    res, xin = [], x
    for l, dl in enumerate(layers):
        if xs is not None:
            xin = xs[l]
        ids = torch.from_numpy(gids[l]).cuda() if ids_given else torch.empty((T, spec.top_k), dtype=torch.int32,
                                                                              device="cuda")
        w = torch.from_numpy(gw[l]).cuda() if ids_given else torch.empty((T, spec.top_k), dtype=torch.float32,
                                                                          device="cuda")
        out = torch.empty((T, spec.d), dtype=torch.float32, device="cuda")
        C.colibri_moe_layer(cfg, xin, dl.Wr, dl.bias, dl.table, dl.shared, ids, w, ids_given, out, ws)
        res.append((out, ids, w))
        xin = out
    torch.cuda.synchronize()
    assert C.colibri_workspace_status(cfg, T, ws) == C.OK
    return [(o.cpu().numpy(), i.cpu().numpy(), ww.cpu().numpy()) for o, i, ww in res]


def run_stack(torch, C, layers, x, ids_given, gids, gw, n_buffers=None, xs=None):
    spec, cfg = layers[0].spec, layers[0].cfg
    T, L = x.shape[0], len(layers)
    ws = torch.empty(C.colibri_moe_stack_workspace_bytes(cfg, T), dtype=torch.uint8, device="cuda")
    nb = n_buffers or L
    outs = [torch.full((T, spec.d), float("nan"), dtype=torch.float32, device="cuda") for _ in range(nb)]
    ids = [torch.from_numpy(gids[l]).cuda() if ids_given else
           torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda") for l in range(L)]
    w = [torch.from_numpy(gw[l]).cuda() if ids_given else
         torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda") for l in range(L)]
    st = [dict(x=None if xs is None else xs[l], Wr=dl.Wr, bias=dl.bias, experts=dl.table, shared=dl.shared,
               ids=ids[l], w=w[l], out=outs[l % nb]) for l, dl in enumerate(layers)]
    C.colibri_moe_stack_decode(cfg, x, st, ids_given, ws)
    torch.cuda.synchronize()
    status = C.colibri_workspace_status(cfg, T, ws)
    return [o.cpu().numpy() for o in outs], [i.cpu().numpy() for i in ids], [v.cpu().numpy() for v in w], status


def bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


@pytest.mark.parametrize("name,T,L,ids_given", [
    ("tiny", 1, 4, False), ("tiny", 5, 3, False), ("tiny", 32, 3, False), ("tiny", 3, 3, True),
    ("tiny_g64", 3, 3, False), ("olmoe_g64", 2, 2, False),
    ("olmoe", 1, 3, False), ("olmoe", 16, 3, False), ("olmoe", 4, 2, True),
    ("glm52", 1, 3, False), ("glm52", 4, 3, False), ("glm52", 1, 2, True),
])
def test_stack_equals_sequential_layers(torch_cuda, C, name, T, L, ids_given):
    torch = torch_cuda
    layers = stack_layers(C, name, L)
    spec = layers[0].spec
    x = torch.from_numpy(synth.activations(spec, 11, T)).cuda()
    gids, gw = given_routing(spec, T, L, 3) if ids_given else (None, None)
    seq = run_sequential(torch, C, layers, x, ids_given, gids, gw)
    outs, ids, w, status = run_stack(torch, C, layers, x, ids_given, gids, gw)
    assert status == C.OK
    for l in range(L):
        assert np.array_equal(ids[l], seq[l][1]), f"layer {l} ids"
        assert np.array_equal(bits(w[l]), bits(seq[l][2])), f"layer {l} weights"
        assert np.array_equal(bits(outs[l]), bits(seq[l][0])), f"layer {l} output"
        assert np.all(np.isfinite(outs[l]))


@pytest.mark.parametrize("name,T,L", [("tiny", 3, 8), ("glm52", 1, 8), ("glm52", 4, 8)])
def test_stack_given_inputs(torch_cuda, C, name, T, L):
    """Every layer with activations of its own (as when attention sits between the MoE
    layers of a model): eight layers in one launch equal eight calls, bit for bit."""
    torch = torch_cuda
    layers = stack_layers(C, name, L)
    spec = layers[0].spec
    xs = [torch.from_numpy(synth.activations(spec, 20 + l, T)).cuda() for l in range(L)]
    seq = run_sequential(torch, C, layers, xs[0], False, None, None, xs=xs)
    outs, ids, w, status = run_stack(torch, C, layers, xs[0], False, None, None, xs=xs)
    assert status == C.OK
    for l in range(L):
        assert np.array_equal(ids[l], seq[l][1]), f"layer {l} ids"
        assert np.array_equal(bits(w[l]), bits(seq[l][2])), f"layer {l} weights"
        assert np.array_equal(bits(outs[l]), bits(seq[l][0])), f"layer {l} output"


def test_stack_two_buffers_in_turn(torch_cuda, C):
    """Layer l writes the buffer layer l - 2 wrote (its input's input): the last two
    outputs still equal the sequential ones."""
    torch = torch_cuda
    L, T = 5, 2
    layers = stack_layers(C, "tiny", L)
    spec = layers[0].spec
    x = torch.from_numpy(synth.activations(spec, 4, T)).cuda()
    seq = run_sequential(torch, C, layers, x, False, None, None)
    outs, ids, _, status = run_stack(torch, C, layers, x, False, None, None, n_buffers=2)
    assert status == C.OK
    assert np.array_equal(bits(outs[(L - 1) % 2]), bits(seq[L - 1][0]))
    assert np.array_equal(bits(outs[(L - 2) % 2]), bits(seq[L - 2][0]))
    for l in range(L):
        assert np.array_equal(ids[l], seq[l][1])


def test_stack_bad_id_stops_and_reports(torch_cuda, C):
    """An out-of-range given id in layer 1 sets the device flag; every CTA stops at the next
    layer boundary and the call returns."""
    torch = torch_cuda
    L, T = 3, 1
    layers = stack_layers(C, "tiny", L)
    spec = layers[0].spec
    gids, gw = given_routing(spec, T, L, 9)
    gids[1, 0, 2] = spec.n_exp
    x = torch.from_numpy(synth.activations(spec, 2, T)).cuda()
    _, _, _, status = run_stack(torch, C, layers, x, True, gids, gw)
    assert status == C.E_DEVICE


def test_stack_argument_checks(torch_cuda, C):
    torch = torch_cuda
    layers = stack_layers(C, "tiny", 3)
    spec, cfg = layers[0].spec, layers[0].cfg
    T = 2
    x = torch.from_numpy(synth.activations(spec, 0, T)).cuda()
    ws = torch.empty(C.colibri_moe_stack_workspace_bytes(cfg, T), dtype=torch.uint8, device="cuda")
    ids = torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda")
    o1 = torch.empty((T, spec.d), dtype=torch.float32, device="cuda")
    o2 = torch.empty_like(o1)

    def lay(dl, out):
        return dict(Wr=dl.Wr, bias=dl.bias, experts=dl.table, shared=dl.shared, ids=ids, w=w, out=out)

    for st, code in [([lay(layers[0], x)], C.E_INVAL),                              # out is the input
                     ([lay(layers[0], o1), lay(layers[1], o1)], C.E_INVAL),         # out is layer 0's
                     ([lay(layers[0], o1)] * (C.STACK_MAX + 1), C.E_INVAL),
                     ([], C.E_INVAL)]:
        with pytest.raises(C.ColibriError) as e:
            C.colibri_moe_stack_decode(cfg, x, st, False, ws)
        assert e.value.status == code
    with pytest.raises(C.ColibriError) as e:
        C.colibri_moe_stack_decode(cfg, x, [lay(layers[0], o1), lay(layers[1], o2)], False, ws[:ws.numel() // 2])
    assert e.value.status == C.E_NOMEM
    torch.cuda.synchronize()
