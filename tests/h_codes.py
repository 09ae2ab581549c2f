"""Checks of the q8(h) codes and scales that the layer leaves in its workspace against
the oracle's, and of the layer output with the slack those codes allow.

Used by the GPU parity tests; its own CPU test (test_h_code_check.py) runs it on
workspaces filled from the oracle."""
import numpy as np

TOL = 2e-3


def ws_slice(ws, off, nbytes, dtype):
    return ws[off:off + nbytes].cpu().numpy().view(dtype)


U32 = 2.0 ** -24  # unit roundoff of fp32


def h_error_bound(orc, v, qx, sx, group=32):
    """[f]: a bound on the relative error of the kernel's fp32 h against the oracle's.

    The kernel adds the d/32 exact 32-column dots times their fp32 scale products (the
    scales of their group of 32 or 64) in fp32 (in any order), so its gate and up are
    within (d/32 + 8) u sum|terms| of the exact sums (the oracle's fp64 sums are exact to
    far below that); relative to h that is the sums' condition kappa = sum|terms| / |sum|,
    the gate's times the condition of silu (1 + |z| sigmoid(-z)), plus a few u for expf,
    the division and the products."""
    ng = qx.shape[0] // 32
    rep = group // 32
    sxg = np.repeat(sx.astype(np.float64), rep)[None, :]
    tg = np.repeat(v["s1"].astype(np.float64), rep, axis=1) * sxg * orc.group_dots(v["w1"], qx)
    tu = np.repeat(v["s3"].astype(np.float64), rep, axis=1) * sxg * orc.group_dots(v["w3"], qx)
    gate, up = tg.sum(1), tu.sum(1)
    kg = np.abs(tg).sum(1) / np.maximum(np.abs(gate), 1e-300)
    ku = np.abs(tu).sum(1) / np.maximum(np.abs(up), 1e-300)
    silu_cond = 1.0 + np.abs(gate) / (1.0 + np.exp(np.clip(gate, -700, 700)))
    return (ng + 8) * U32 * (kg * silu_cond + ku) + 8 * U32


def bf16_codes(raw):
    """[rows][f] integer codes from the prefill's bf16 h codes (inside each run of 8,
    element k at 2*(k%4) + k/4)."""
    k = np.arange(raw.shape[1])
    pos = (k & ~7) + ((k & 3) << 1) + ((k >> 2) & 1)
    return (raw[:, pos].astype(np.uint32) << 16).view(np.float32).astype(np.int64)


def check_h_codes_and_output(orc, C, spec, host, x, ids, w, ws, out, ref, tol=TOL, tokens=None, threads=1):
    """q8(h) codes and scales of every (token, expert) pair against the oracle's, then
    the layer output. Returns the number of codes that differ.

    x, ids, w: the whole batch the layer ran on (T tokens). tokens: the token indices to
    check (default all T); out and ref then hold those tokens' rows, in that order (ref
    from the oracle on those tokens). threads > 1 checks tokens in parallel (the oracle's
    C calls release the GIL).

    Codes and scales must be equal, except where the oracle's h lies within the kernel's
    fp32 error (h_error_bound) of a rounding boundary of q8: there either code is a
    correct rounding of h, so the kernel's may differ by one (and a group's scale by the
    largest error of a |h| of the group, over 127). The output must be within tol * rms(oracle), plus, for each
    token, the most its differing h codes and scales can move it: the pair's weight times
    |W2| (dequantised) applied to |h_kernel - h_oracle| (dequantised). Where every code
    agrees that extra term is zero."""
    T, K, d = x.shape[0], spec.top_k, spec.d
    gq = getattr(spec, "group", 32)
    tokens = list(range(T)) if tokens is None else [int(t) for t in tokens]
    v = C.colibri_moe_workspace_view(C.layer_cfg(spec), T)
    rows = T * K + (T if spec.has_shared else 0)
    if T > 32:
        codes = bf16_codes(ws_slice(ws, v.hbf, 2 * rows * v.fmax, np.uint16).reshape(rows, v.fmax))
    else:
        codes = ws_slice(ws, v.hq, rows * v.fmax, np.int8).reshape(rows, v.fmax).astype(np.int64)
    scales = ws_slice(ws, v.hs, 4 * rows * v.hs_stride, np.float32).reshape(rows, v.hs_stride)
    qx, sx = orc.q8_quantize(x[tokens], group=gq)

    def one(j):
        t = tokens[j]
        allow = np.zeros(d)
        n_diff = 0
        pairs = [(t * K + i, host.expert(int(ids[t, i])), float(w[t, i]), spec.ffn) for i in range(K)]
        if spec.has_shared:
            pairs.append((T * K + t, host.shared(), 1.0, spec.shared_ffn))
        for pr, view, wt, f in pairs:
            _, qh, sh, h = orc.expert_token(view, qx[j], sx[j], want_h=True, group=gq)
            c, gsc = codes[pr, :f], scales[pr, :f // gq]
            dq = c - qh
            dsc = gsc.view(np.uint32) != sh.view(np.uint32)
            if not (dq.any() or dsc.any()):
                continue
            assert np.abs(dq).max() <= 1, (t, pr)
            relg = h_error_bound(orc, view, qx[j], sx[j], gq).reshape(-1, gq)
            sh64 = sh.astype(np.float64)
            assert np.all(sh64 > 0), (t, pr)
            r = np.abs(h.astype(np.float64)).reshape(-1, gq) / sh64[:, None]
            # the scale amax / 127 moves by at most the largest error of a |h| of the group
            rel_scale = (relg * r).max(1) / 127.0 + 2 * U32
            assert np.all(np.abs(gsc / sh64 - 1.0) <= rel_scale), (t, pr)
            window = (relg + rel_scale[:, None]) * r
            ambiguous = (np.abs(r - np.floor(r) - 0.5) <= window).ravel()
            assert np.all(ambiguous[dq != 0]), (t, pr, np.flatnonzero(dq)[:4])
            n_diff += int(np.count_nonzero(dq))
            dh = np.abs(c * np.repeat(gsc.astype(np.float64), gq) - qh * np.repeat(sh64, gq))
            w2 = np.abs(orc.unpack_int4(view["w2"]).astype(np.float64))
            w2 *= np.repeat(view["s2"].astype(np.float64), gq, axis=1)
            allow += wt * (w2 @ dh)
        return allow, n_diff

    if threads > 1 and len(tokens) > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(threads) as ex:
            res = list(ex.map(one, range(len(tokens))))
    else:
        res = [one(j) for j in range(len(tokens))]
    allow = np.stack([a for a, _ in res]) if res else np.zeros((0, d))
    n_diff = sum(n for _, n in res)
    want = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(want ** 2))
    err = np.abs(np.asarray(out, np.float64) - want)
    bad = err > tol * rms + allow * (1 + 1e-6)
    assert not bad.any(), (f"{int(bad.sum())} outputs off; worst excess "
                           f"{float((err - tol * rms - allow).max()):.3e} (rms {rms:.3e})")
    return n_diff


def h_codes_checked(spec, n_tokens):
    """Codes of q8(h) that check_h_codes_and_output compares for n_tokens tokens."""
    return n_tokens * (spec.top_k * spec.ffn + (spec.shared_ffn if spec.has_shared else 0))
