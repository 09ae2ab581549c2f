"""The q8(h) checker of the GPU parity tests, run on CPU on workspaces filled from the
oracle: it must accept the oracle's own codes, reject a code changed away from a
rounding boundary, and accept a change at an ambiguous position only with the output
moved no further than that change explains. No kernel runs here."""
import numpy as np
import pytest

from routed_expert_ffn_grouped_b300 import build as cbuild
from routed_expert_ffn_grouped_b300 import colibri as C
from routed_expert_ffn_grouped_b300 import synth

from h_codes import U32, check_h_codes_and_output, h_error_bound

torch = pytest.importorskip("torch")

SMALL = synth.TINY.replace(name="hcheck", d=256, ffn=128, n_exp=8, top_k=8, n_group=1, topk_group=1,
                           shared_ffn=128)


@pytest.fixture(scope="module")
def lib():
    cbuild.build()
    return C.lib()


def oracle_workspace(orc, spec, host, x, ids, plant=None):
    """A workspace holding the oracle's q8(h) codes and scales where the layer keeps its
    own (decode: int8 codes; prefill: bf16 codes in the tensor-core order). plant =
    (pair row, column, delta) changes one code."""
    T, K = x.shape[0], spec.top_k
    cfg = C.layer_cfg(spec)
    v = C.colibri_moe_workspace_view(cfg, T)
    ws = np.zeros(C.colibri_moe_workspace_bytes(cfg, T), np.uint8)
    rows = T * K + (T if spec.has_shared else 0)
    hq = np.zeros((rows, v.fmax), np.int8)
    hs = np.zeros((rows, v.hs_stride), np.float32)
    qx, sx = orc.q8_quantize(x)
    for t in range(T):
        pairs = [(t * K + i, host.expert(int(ids[t, i])), spec.ffn) for i in range(K)]
        if spec.has_shared:
            pairs.append((T * K + t, host.shared(), spec.shared_ffn))
        for pr, view, f in pairs:
            _, qh, sh = orc.expert_token(view, qx[t], sx[t])
            hq[pr, :f], hs[pr, :f // 32] = qh, sh
    if plant is not None:
        hq[plant[0], plant[1]] += plant[2]
    if T > 32:
        k = np.arange(v.fmax)
        pos = (k & ~7) + ((k & 3) << 1) + ((k >> 2) & 1)
        raw = np.zeros((rows, v.fmax), np.uint16)
        raw[:, pos] = (hq.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        ws[v.hbf:v.hbf + raw.nbytes] = raw.view(np.uint8).ravel()
    else:
        ws[v.hq:v.hq + hq.nbytes] = hq.view(np.uint8).ravel()
    ws[v.hs:v.hs + hs.nbytes] = hs.view(np.uint8).ravel()
    return torch.from_numpy(ws)


def boundary_positions(orc, spec, host, x, ids):
    """Over every (token, pair): the h code nearest a rounding boundary relative to the
    kernel's error window, as (token, pair row, column, inside the window, the code's
    other rounding), and the code of token 0's first pair farthest from a boundary, as
    (pair row, column, a change of one step)."""
    T, K = x.shape[0], spec.top_k
    qx, sx = orc.q8_quantize(x)
    best, far = None, None
    for t in range(T):
        pairs = [(t * K + i, host.expert(int(ids[t, i]))) for i in range(K)]
        for pr, view in pairs:
            _, qh, sh, h = orc.expert_token(view, qx[t], sx[t], want_h=True)
            relg = h_error_bound(orc, view, qx[t], sx[t]).reshape(-1, 32)
            r = np.abs(h.astype(np.float64)).reshape(-1, 32) / sh.astype(np.float64)[:, None]
            window = ((relg + ((relg * r).max(1) / 127.0 + 2 * U32)[:, None]) * r).ravel()
            frac = (r - np.floor(r)).ravel()
            dist = np.abs(frac - 0.5)
            j = int(np.argmin(dist - window))
            if best is None or dist[j] - window[j] < best[0]:
                # the other rounding: one step further from zero if q8 rounded |h| down
                other = int(np.sign(h[j])) * (1 if frac[j] < 0.5 else -1)
                best = (dist[j] - window[j], t, pr, j, bool(dist[j] <= window[j]), other)
            if far is None:
                jf = int(np.argmax(dist))
                far = (pr, jf, 1 if qh[jf] < 127 else -1)
    return best[1:], far


@pytest.mark.parametrize("T", [3, 40])  # decode and prefill workspace layouts
def test_checker_on_oracle_workspaces(lib, orc, T):
    host = synth.make_layer(SMALL, 0)
    x = synth.activations(SMALL, 0, T, step=5)
    ref, ids, w = orc.moe_layer(SMALL, x, host.Wr, host.bias, host.expert, host.shared())
    # the oracle's own codes: nothing differs, the plain tolerance holds
    ws = oracle_workspace(orc, SMALL, host, x, ids)
    assert check_h_codes_and_output(orc, C, SMALL, host, x, ids, w, ws, ref, ref) == 0
    rms = np.sqrt(np.mean(ref.astype(np.float64) ** 2))
    moved = ref.copy()
    moved[0, 0] += np.float32(3e-3 * rms)
    with pytest.raises(AssertionError):
        check_h_codes_and_output(orc, C, SMALL, host, x, ids, w, ws, moved, ref)
    (t_amb, pr_amb, j_amb, amb_ok, other), (pr_far, j_far, step) = boundary_positions(orc, SMALL, host, x, ids)
    # a code changed far from any boundary is an error, whatever the output
    ws_far = oracle_workspace(orc, SMALL, host, x, ids, plant=(pr_far, j_far, step))
    with pytest.raises(AssertionError):
        check_h_codes_and_output(orc, C, SMALL, host, x, ids, w, ws_far, ref, ref)
    # two steps away from the oracle's code is an error even at a boundary
    ws_two = oracle_workspace(orc, SMALL, host, x, ids, plant=(pr_amb, j_amb, 2 * other))
    with pytest.raises(AssertionError):
        check_h_codes_and_output(orc, C, SMALL, host, x, ids, w, ws_two, ref, ref)
    assert amb_ok, "no h code of this batch lies at a rounding boundary"
    # at an ambiguous position the other rounding is accepted; the output may move by what
    # that code explains, but another token's output may not move at all
    ws_amb = oracle_workspace(orc, SMALL, host, x, ids, plant=(pr_amb, j_amb, other))
    assert check_h_codes_and_output(orc, C, SMALL, host, x, ids, w, ws_amb, ref, ref) == 1
    elsewhere = ref.copy()
    elsewhere[(t_amb + 1) % T, 0] += np.float32(3e-3 * rms)
    with pytest.raises(AssertionError):
        check_h_codes_and_output(orc, C, SMALL, host, x, ids, w, ws_amb, elsewhere, ref)
