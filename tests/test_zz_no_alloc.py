"""colibri_moe_layer_noalloc against colibri_moe_layer, through the C ABI.

The no-allocation entry point is for callers that cannot allocate device memory when
they run the layer (a runtime that owns all device memory through its own pool, a
plugin handed only its inputs and outputs, a loop that cannot afford cudaMalloc's
implicit device synchronisation). It runs the same layer on a fixed scratch array that
the library holds in device memory. Two calls in a row, on different inputs, must each
give what colibri_moe_layer gives on a caller-allocated workspace, within the layer
tolerance of the parity tests (max |err| <= 2e-3 * rms). The second call also shows that
what the first call left in the shared scratch does not leak into the next result.

This file is collected last so that a run stopping at its first failure has already
run every other test. It needs nothing from the other test modules.
"""
import numpy as np
import pytest

from routed_expert_ffn_grouped_b300 import synth

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


def _rms_err(got, want):
    want = np.asarray(want, np.float64)
    rms = float(np.sqrt(np.mean(want ** 2)))
    err = float(np.max(np.abs(np.asarray(got, np.float64) - want)))
    return err, rms


_layers = {}


def _device_layer(C, spec):
    if spec.name not in _layers:
        _layers[spec.name] = C.DeviceLayer(synth.make_layer(spec, 0))
    return _layers[spec.name]


# GLM-5.2-shaped at T = 32: the largest batch of that layer whose workspace fits the
# fixed scratch array
@pytest.mark.parametrize("name,T", [("tiny", 4), ("olmoe", 16), ("glm52", 32)])
def test_noalloc_matches_workspace_entry_point(torch_cuda, C, name, T):
    torch = torch_cuda
    spec = synth.SPECS[name]
    dl = _device_layer(C, spec)
    cfg = dl.cfg
    assert C.colibri_moe_workspace_bytes(cfg, T) <= C.NOALLOC_SCRATCH_BYTES

    def buffers():
        return (torch.empty((T, spec.d), dtype=torch.float32, device="cuda"),
                torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda"),
                torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda"))

    ws = torch.empty(C.colibri_moe_workspace_bytes(cfg, T), dtype=torch.uint8, device="cuda")
    for call in range(2):                       # two calls in a row, different tokens
        x = torch.from_numpy(synth.activations(spec, 0, T, step=100 + call)).cuda()
        out_a, ids_a, w_a = buffers()
        C.colibri_moe_layer(cfg, x, dl.Wr, dl.bias, dl.table, dl.shared, ids_a, w_a, False, out_a, ws)
        out_b, ids_b, w_b = buffers()
        out_b.fill_(float("nan"))
        C.colibri_moe_layer_noalloc(cfg, x, dl.Wr, dl.bias, dl.table, dl.shared, ids_b, w_b, False, out_b)
        torch.cuda.synchronize()
        assert C.colibri_workspace_status(cfg, T, ws) == C.OK
        assert np.array_equal(ids_b.cpu().numpy(), ids_a.cpu().numpy()), f"call {call}: ids differ"
        np.testing.assert_allclose(w_b.cpu().numpy(), w_a.cpu().numpy(), rtol=1e-6, atol=0)
        err, rms = _rms_err(out_b.cpu().numpy(), out_a.cpu().numpy())
        assert err <= TOL * rms, f"call {call}: max err {err:.3e} > {TOL} * rms {rms:.3e}"


def test_noalloc_rejects_oversized_batches(torch_cuda, C):
    """A batch whose workspace exceeds the fixed scratch is refused before any launch."""
    spec = synth.GLM52
    cfg = C.layer_cfg(spec)
    T = 1
    while C.colibri_moe_workspace_bytes(cfg, T) <= C.NOALLOC_SCRATCH_BYTES:
        T *= 2
    assert T > 32                               # the documented limit: up to T = 32 fits
    x = np.zeros((T, spec.d), np.float32)       # host arrays: nothing may be touched
    with pytest.raises(C.ColibriError) as e:
        C.colibri_moe_layer_noalloc(cfg, x, x, None, x, None, x, x, True, x, stream=0)
    assert e.value.status == C.E_NOMEM
