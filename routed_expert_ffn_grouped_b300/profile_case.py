"""A GLM-5.2-shaped layer with only the experts it routes to resident, for profiling.

    python -m routed_expert_ffn_grouped_b300.profile_case decode  [--T 1] [--iters 5] [--f32]
    python -m routed_expert_ffn_grouped_b300.profile_case prefill [--T 512] [--experts 32] [--iters 3]

Each token is given 8 distinct experts out of a fixed set (ids passed in, the router
skipped), so the device holds only those experts (plus the shared one): the decode case
streams exactly the bytes of one decode step of the full layer (8 routed experts per
token and the shared expert), with a few hundred MB on the device instead of 6 GB. Runs
`--iters` layer calls, printing each call's time (CUDA events) and the device status.
`--f32` runs the decode layer on fp32 activations (colibri_moe_layer_f32) instead.
"""
from __future__ import annotations

import argparse

import numpy as np


def main():
    import torch

    from . import build, synth
    from . import colibri as C

    p = argparse.ArgumentParser()
    p.add_argument("mode", choices=["decode", "prefill"])
    p.add_argument("--T", type=int, default=None)
    p.add_argument("--experts", type=int, default=None, help="resident routed experts (prefill)")
    p.add_argument("--iters", type=int, default=5)
    p.add_argument("--f32", action="store_true", help="decode on fp32 activations")
    a = p.parse_args()
    build.build()
    spec = synth.GLM52
    T = a.T or (1 if a.mode == "decode" else 512)
    n_used = a.experts or (min(spec.n_exp, 8 * T) if a.mode == "decode" else 32)
    rng = np.random.default_rng(0)
    used = sorted(rng.choice(spec.n_exp, size=n_used, replace=False).tolist())
    lay = C.colibri_blob_layout_for(spec.d, spec.ffn)
    blobs = torch.empty((n_used, lay.nbytes), dtype=torch.uint8, device="cuda")
    table = (C.Expert * spec.n_exp)()
    for k, e in enumerate(used):
        blobs[k].copy_(torch.from_numpy(synth.expert_blob(spec, 0, 0, e)))
        b = blobs[k].data_ptr()
        table[e] = C.Expert(b + lay.w1, b + lay.w3, b + lay.w2, b + lay.s1, b + lay.s3, b + lay.s2)
    tdev = torch.frombuffer(bytearray(bytes(table)), dtype=torch.uint8).cuda()
    shb = torch.from_numpy(synth.expert_blob(spec, 0, 0, 0, shared=True)).cuda()
    sl = C.colibri_blob_layout_for(spec.d, spec.shared_ffn)
    b = shb.data_ptr()
    shared = C.Expert(b + sl.w1, b + sl.w3, b + sl.w2, b + sl.s1, b + sl.s3, b + sl.s2)
    cfg = C.layer_cfg(spec)
    if a.mode == "decode" and n_used >= 8 * T:
        ids = np.array(used[:8 * T], np.int32).reshape(T, 8)
    else:
        ids = np.stack([rng.choice(used, size=8, replace=False) for _ in range(T)]).astype(np.int32)
    idsd = torch.from_numpy(ids).cuda()
    w = torch.full((T, 8), 0.3, dtype=torch.float32, device="cuda")
    x = torch.from_numpy(synth.activations(spec, 0, T)).cuda()
    out = torch.empty((T, spec.d), dtype=torch.float32, device="cuda")
    f32 = a.f32 and a.mode == "decode"
    ws_bytes = (C.colibri_moe_f32_workspace_bytes if f32 else C.colibri_moe_workspace_bytes)(cfg, T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    layer = C.colibri_moe_layer_f32 if f32 else C.colibri_moe_layer
    st, en = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(a.iters):
        st.record()
        layer(cfg, x, None, None, tdev, shared, idsd, w, True, out, ws)
        en.record()
        torch.cuda.synchronize()
        print(f"call {i}: {st.elapsed_time(en) * 1e3:.1f} us")
    print("device status", C.colibri_workspace_status(cfg, T, ws))


if __name__ == "__main__":
    main()
