"""64-element quantisation groups (the pages' int4 containers: aifrontierpost tutorial,
"Step 3 -- Get a model") on the CUDA path, against the oracle's 64-group layer.

The same bars as the 32-group parity tests: q8 codes and scales, expert ids, bucket lists
bit-exact; routing weights within 1e-6; every q8(h) code equal to the oracle's except at a
provable rounding ambiguity (then one step), and outputs within 2e-3 * rms(oracle) plus
the effect of such codes. Decode (in-kernel routing, the q8 of h over two gate/up items),
prefill (tcgen05 grouped GEMMs, the q8 of h across two epilogue warps) and the
fp32-activation decode.
"""
import numpy as np
import pytest

from routed_expert_ffn_grouped_b300 import synth

from h_codes import check_h_codes_and_output, h_codes_checked
from test_gpu_parity import (assert_buckets_exact, assert_rms_close, dev_layer, run_layer, run_layer_f32,
                             to_dev, ws_slice)

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


@pytest.mark.parametrize("rows,cols", [(1, 512), (4, 6144), (2048, 6144), (3, 64)])
def test_q8_g64_bit_exact(torch_cuda, C, orc, rows, cols):
    torch = torch_cuda
    rng = np.random.default_rng(rows * 13 + cols)
    x = (rng.standard_normal((rows, cols)) * rng.uniform(0.01, 50, (rows, 1))).astype(np.float32)
    x[0, :64] = 0.0                                            # an all-zero group
    g = 64 if cols >= 128 else 0
    x[-1, g:g + 64] = (np.arange(64, dtype=np.float32) - 31.5) * 2   # half-steps after scaling
    q = torch.empty((rows, cols), dtype=torch.int8, device="cuda")
    s = torch.empty((rows, cols // 64), dtype=torch.float32, device="cuda")
    C.colibri_q8_quantize(to_dev(torch, x), q, s, group=64)
    torch.cuda.synchronize()
    qo, so = orc.q8_quantize(x, group=64)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))


def _check_layer(torch, C, orc, flip_report, spec, T, row_scale=False, step=41):
    host, dl = dev_layer(C, spec)
    x = synth.activations(spec, 0, T, step=step, row_scale=row_scale)
    out, ids, w, ws = run_layer(torch, C, dl, x)
    assert C.colibri_workspace_status(dl.cfg, T, ws) == C.OK
    ref, ids_o, w_o = orc.moe_layer(spec, x, host.Wr, host.bias, host.expert, host.shared(), group=64)
    assert np.array_equal(ids, ids_o)
    np.testing.assert_allclose(w, w_o, rtol=1e-6)
    assert_rms_close(out, ref)
    v = C.colibri_moe_workspace_view(dl.cfg, T)
    qx = ws_slice(ws, v.qx, T * spec.d, np.int8).reshape(T, spec.d)
    sx = ws_slice(ws, v.sx, 4 * T * spec.d // 64, np.float32).reshape(T, -1)
    qo, so = orc.q8_quantize(x, group=64)
    assert np.array_equal(qx, qo) and np.array_equal(sx.view(np.uint32), so.view(np.uint32))
    assert_buckets_exact(C, dl, ws, T, ids_o)
    n = check_h_codes_and_output(orc, C, spec, host, x, ids_o, w_o, ws, out, ref)
    flip_report(n, h_codes_checked(spec, T))


@pytest.mark.parametrize("name,T", [("tiny_g64", 1), ("tiny_g64", 4), ("tiny_g64", 13), ("olmoe_g64", 1),
                                    ("olmoe_g64", 16), ("glm52_g64", 1), ("glm52_g64", 4)])
def test_g64_decode_parity(torch_cuda, C, orc, flip_report, name, T):
    """Decode at 64-element groups: the q8 of h spans two 32-row gate/up items, and the one
    that finishes second quantises both halves."""
    _check_layer(torch_cuda, C, orc, flip_report, synth.SPECS[name], T)


@pytest.mark.parametrize("name,T", [("tiny_g64", 33), ("tiny_g64", 100), ("olmoe_g64", 48)])
def test_g64_prefill_parity(torch_cuda, C, orc, flip_report, name, T):
    """Prefill at 64-element groups: one scale pair per two 32-column MMA steps, and the
    q8 of h across the two epilogue warps that hold each 64-row group."""
    _check_layer(torch_cuda, C, orc, flip_report, synth.SPECS[name], T, row_scale=True, step=43)


def test_g64_glm_prefill_sampled(torch_cuda, C, orc, flip_report):
    """The GLM-shaped prefill (T = 2048) at 64-element groups: ids, weights and bucket lists
    of the whole batch, outputs and q8(h) codes of 48 tokens (the busiest expert's last
    tile among them)."""
    torch = torch_cuda
    spec = synth.GLM52_64
    host, dl = dev_layer(C, spec)
    T, K = 2048, spec.top_k
    x = synth.activations(spec, 0, T, step=47, row_scale=True)
    out, ids, w, ws = run_layer(torch, C, dl, x)
    assert C.colibri_workspace_status(dl.cfg, T, ws) == C.OK
    io_all, wo_all = orc.router_topk(spec, x, host.Wr, host.bias)
    assert np.array_equal(ids, io_all)
    np.testing.assert_allclose(w, wo_all, rtol=1e-6)
    off_o, pairs_o = assert_buckets_exact(C, dl, ws, T, io_all)
    counts = np.bincount(io_all.ravel(), minlength=spec.n_exp)
    e = int(np.argmax(counts))
    last = int(off_o[e]) + ((int(counts[e]) - 1) // 64) * 64
    toks = set(int(p) // K for p in pairs_o[last:int(off_o[e]) + int(counts[e])])
    toks.update(int(t) for t in np.random.default_rng(9).choice(T, 40, replace=False))
    toks = sorted(toks)
    ref, _, _ = orc.moe_layer(spec, x[toks], host.Wr, host.bias, host.expert, host.shared(), group=64)
    n = check_h_codes_and_output(orc, C, spec, host, x, io_all, wo_all, ws, out[toks], ref, tokens=toks,
                                 threads=8)
    flip_report(n, h_codes_checked(spec, len(toks)))


@pytest.mark.parametrize("name,T", [("tiny_g64", 1), ("tiny_g64", 13), ("glm52_g64", 1), ("glm52_g64", 4)])
def test_g64_f32_parity(torch_cuda, C, orc, name, T):
    """The fp32-activation decode with 64-element weight groups."""
    torch = torch_cuda
    spec = synth.SPECS[name]
    host, dl = dev_layer(C, spec)
    x = synth.activations(spec, 0, T, step=17)
    out, ids, w, ws = run_layer_f32(torch, C, dl, x)
    assert C.colibri_workspace_status(dl.cfg, T, ws) == C.OK
    ref, ids_o, w_o = orc.moe_layer(spec, x, host.Wr, host.bias, host.expert, host.shared(), act="f32", group=64)
    assert np.array_equal(ids, ids_o)
    np.testing.assert_allclose(w, w_o, rtol=1e-6)
    assert_rms_close(out, ref)


def test_g64_ids_given(torch_cuda, C, orc):
    torch = torch_cuda
    spec = synth.GLM52_64
    host, dl = dev_layer(C, spec)
    ids, w = synth.streaming_ids(spec, 5, 1, 2)
    ids, w = ids[:, 0], w[:, 0]
    x = synth.activations(spec, 5, 2)
    out, ids_d, _, ws = run_layer(torch, C, dl, x, ids, w)
    assert C.colibri_workspace_status(dl.cfg, 2, ws) == C.OK
    ref, _, _ = orc.moe_layer(spec, x, None, None, host.expert, host.shared(), ids=ids, w=w, group=64)
    assert_rms_close(out, ref)
