#!/usr/bin/env python3
"""Benchmark of one routed MoE FFN layer on B300 (GLM-5.2-shaped decode by default).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl colibri|reference]
                    [--workload glm52_decode_t1|glm52_decode_t4|olmoe_decode_t1|...]

A step is one pass of the whole layer (q8, router, bucketing, gate/up, down, combine)
over one batch of T synthetic tokens, with all experts resident in HBM. Each timed step
is one CUDA-graph replay bracketed by CUDA events on the launching stream; between
steps (outside the events) the next token's activations are copied in, a 256 MB buffer
is written to flush the 126 MB L2, a second 256 MB buffer is read (no dirty lines left to
write back), and the layer before runs once: a layer of the same shape with its own
weights at other addresses, as in a model where layers run back to back. So the timed
step starts with none of its own data in L2 but with the kernels' code warm. Prints one
JSON line.

--impl reference times the CPU oracle (plain C, one core) on the same workload: each
step is one expert pass of one token (the router and the shared expert ride with the
first of a token's passes), so the step count of the GPU arm stays affordable.

Multi-GPU (torchrun): the layer does not shard here, so N ranks run N independent
replicas (weak scaling); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from routed_expert_ffn_grouped_b300 import synth  # noqa: E402

METRIC = "MoE-layer decode tokens/s; expert-weight HBM GB/s as % of B300 peak"
WORKLOADS = {
    "glm52_decode_t1": ("glm52", 1, False),
    "glm52_decode_t4": ("glm52", 4, False),
    "olmoe_decode_t1": ("olmoe", 1, False),
    "olmoe_decode_t16": ("olmoe", 16, False),
    "glm52_prefill_t2048": ("glm52", 2048, True),
    "glm52_stream_8l": ("glm52", 1, False),
    # the decode variant on fp32 activations (colibri_moe_layer_f32)
    "glm52_decode_t1_f32": ("glm52", 1, False),
    "glm52_decode_t4_f32": ("glm52", 4, False),
    # the same GLM-shaped layer with the 64-element groups of the pages' int4 containers
    "glm52_decode_t1_g64": ("glm52_g64", 1, False),
    "glm52_decode_t4_g64": ("glm52_g64", 4, False),
    "glm52_prefill_t2048_g64": ("glm52_g64", 2048, True),
    # eight resident GLM-shaped layers in one launch (colibri_moe_stack_decode)
    "glm52_decode_t1_stack8": ("glm52", 1, False),
    "glm52_decode_t4_stack8": ("glm52", 4, False),
    "olmoe_decode_t1_stack8": ("olmoe", 1, False),
}
STACK_LAYERS = 8
DEFAULT_WORKLOAD = "glm52_decode_t1"
N_X = 64                 # distinct activation batches cycled through
L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="colibri", choices=["colibri", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--hot-slots", type=int, default=0,
                   help="glm52_stream_8l: cache slots held by the most used experts (0: plain LRU)")
    p.add_argument("--cache-sim", action="store_true",
                   help="glm52_stream_8l: hit rates of the cache policy for several hot-set sizes, "
                        "simulated on the host (no GPU)")
    p.add_argument("--predictor", default="previous", choices=["previous", "lookahead"],
                   help="expert streaming: next-layer prefetch from an emulated router lookahead "
                        "that names each true id with probability 0.716, or the previous step's ids")
    p.add_argument("--prefetch-chunk-mb", type=float, default=1.0,
                   help="expert streaming: prefetch chunk size (queued, cancellable prefetch); "
                        "0: whole-blob prefetch copies enqueued at once")
    p.add_argument("--prefetch-inflight", type=int, default=2,
                   help="expert streaming: prefetch chunks (or whole blobs) in flight at most")
    p.add_argument("--ids-ahead", action="store_true",
                   help="expert streaming: the host knows every layer's ids before the step starts "
                        "(no wait for the previous layer before a lookup)")
    return p.parse_args()


# ---------------------------------------------------------------- helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def traffic_from_profiles(summary: str, source: str, workload: str):
    """dram bytes per launch recorded by ncu in profiles/<summary>.md for `workload`, or
    None when there is none or the kernel source changed since (the summary stores the
    sha256 of the source file it measured)."""
    path = os.path.join(ROOT, "profiles", f"{summary}.md")
    src = os.path.join(ROOT, "routed_expert_ffn_grouped_b300", "csrc", source)
    try:
        text = open(path).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    m = re.search(rf"traffic_bytes_per_launch\[{workload}\]:\s*([0-9.e+]+)", text)
    s = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != sha:
        return None
    return float(m.group(1))


class ClockSampler:
    """Samples SM clocks and clock-event reasons with `nvidia-smi -lms` while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, torch, device_index: int, period_ms: int = 20):
        import subprocess
        self.subprocess = subprocess
        self.period = period_ms
        self.index = device_index
        try:
            bus = torch.cuda.get_device_properties(device_index).pci_bus_id
            self.sel = ["--id=" + bus] if bus else []
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            first = vis.split(",")[device_index] if vis else str(device_index)
            self.sel = ["--id=" + first]
        self.lines = []
        self.first = []

    def __enter__(self):
        try:
            self.proc = self.subprocess.Popen(
                ["nvidia-smi", *self.sel, "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 f"-lms={self.period}"], stdout=self.subprocess.PIPE, stderr=self.subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        # the first sample marks that the sampler runs before the timed region starts
        first = self.proc.stdout.readline()
        self.first = [first] if first.strip() else []
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = self.first + [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(torch):
    """World, rank and local rank from the launcher's environment; for N > 1 one process
    group over all ranks (NCCL with GPUs, gloo without)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    gpu = torch.cuda.is_available()
    if world > 1:
        import torch.distributed as dist
        if gpu:
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if gpu else "gloo")
    elif gpu:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(torch, world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(torch, world, v: float) -> float:
    """The largest v over the ranks (every rank gets it)."""
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(world: int, tokens_per_rank: int, steps: int, max_ms: float) -> float:
    """Whole-job tokens/s: every rank runs its own replica of the layer on its own tokens,
    so the job processes world x tokens_per_rank x steps tokens in the slowest rank's time."""
    return world * tokens_per_rank * steps / (max_ms / 1e3)


def blob_bytes(spec, f):
    gq = getattr(spec, "group", 32)
    L = synth.blob_layout(spec.d, f, gq)
    gate_up = 2 * (f * spec.d // 2) + 2 * 4 * f * (spec.d // gq)
    down = spec.d * f // 2 + 4 * spec.d * (f // gq)
    return L.nbytes, gate_up, down


# ---------------------------------------------------------------- oracle timing
def expert_load(ids_steps: np.ndarray, n_exp: int) -> dict:
    """How the routed pairs of each timed step's batch spread over the experts, averaged
    over the steps: distinct experts, the busiest expert's tokens, that over the mean per
    expert, and percentiles of tokens per expert (all E experts, zeros included).
    ids_steps: [steps][T][top_k]."""
    steps = ids_steps.shape[0]
    counts = np.stack([np.bincount(ids_steps[i].ravel(), minlength=n_exp) for i in range(steps)])
    pairs = counts.sum(1)
    mean = pairs / n_exp
    return {"steps": int(steps), "pairs_per_step": float(pairs.mean()),
            "distinct_experts": float((counts > 0).sum(1).mean()),
            "max_tokens_per_expert": float(counts.max(1).mean()),
            "max_over_mean": float((counts.max(1) / mean).mean()),
            "tokens_per_expert_p50_p90_p99": [float(np.percentile(counts, q)) for q in (50, 90, 99)]}


def host_info() -> dict:
    """The bench host's CPU: logical cores and model name."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"nproc": os.cpu_count(), "cpu_model": model}


def informational(fn, *args) -> dict:
    """fn(*args), or the error it raised: an informational field never stops the bench."""
    try:
        return fn(*args)
    except Exception as e:  # noqa: BLE001
        return {"error": f"{type(e).__name__}: {e}"}


def is_f32(workload: str) -> bool:
    return workload.endswith("_f32")


def oracle_tokens_per_s(spec, host, xs, budget_s: float, max_tokens: int, act: str = "q8"):
    import oracle
    oracle.lib()
    t0 = time.perf_counter()
    n = 0
    while n < max_tokens:
        oracle.moe_layer(spec, xs[n % len(xs)], host.Wr, host.bias, host.expert, host.shared(), act=act,
                         group=getattr(spec, "group", 32))
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return n / dt, n, dt


def oracle_tokens_per_s_all_cores(spec, host, xs, budget_s: float, act: str = "q8"):
    """The oracle as it stands on every host core: one token per call, as many calls in
    flight as the host has logical cores (host threads; the oracle's C calls release the
    GIL, and tokens are independent). Returns (tokens/s, tokens, seconds, threads)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    oracle.lib()
    threads = max(1, os.cpu_count() or 1)
    gq = getattr(spec, "group", 32)
    stop = time.perf_counter() + budget_s
    counts = [0] * threads

    def worker(k):
        i = k
        while time.perf_counter() < stop:
            x = xs[i % len(xs)]
            oracle.moe_layer(spec, x[None] if x.ndim == 1 else x[:1], host.Wr, host.bias, host.expert,
                             host.shared(), act=act, group=gq)
            counts[k] += 1
            i += threads
    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(worker, range(threads)))
    dt = time.perf_counter() - t0
    n = sum(counts)
    return n / dt, n, dt, threads


def run_reference(args):
    """The oracle on the host cores, step = one expert pass of one token."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.lib()
    name, T, row_scale = WORKLOADS[args.workload]
    spec = synth.SPECS[name]
    host = synth.make_layer(spec, args.seed)
    xs = [synth.activations(spec, args.seed, 1, step=i, row_scale=row_scale)[0] for i in range(N_X)]
    per_tok = spec.top_k + (1 if spec.has_shared else 0)
    state = {"tok": -1}
    f32 = is_f32(args.workload)
    gq = getattr(spec, "group", 32)

    def expert(views):
        if f32:
            return oracle.expert_token_f32(views, state["x"])[0]
        return oracle.expert_token(views, state["q"], state["s"], group=gq)[0]

    def step(i):
        t, slot = divmod(i, per_tok)
        x = xs[t % N_X]
        if slot == 0 or state["tok"] != t:
            q, s = oracle.q8_quantize(x, group=gq)
            ids, w = oracle.router_topk(spec, x[None], host.Wr, host.bias)
            state.update(tok=t, x=x, q=q, s=s, ids=ids[0], w=w[0], acc=np.zeros(spec.d))
        if spec.has_shared and slot == per_tok - 1:
            state["acc"] += expert(host.shared())
        elif slot < spec.top_k:
            state["acc"] += float(state["w"][slot]) * expert(host.expert(int(state["ids"][slot])))

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = (args.steps / per_tok) / dt       # tokens/s: one token per per_tok steps
    sample = (f"{args.steps} steps = {args.steps / per_tok:.1f} tokens of the {args.workload} layer, "
              f"one expert pass of one token per step, single-threaded C oracle")
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "i4 x f32 -> f64" if f32 else "i8xi4->i32, f64",
            "data": "synthetic", "config": workload_config(spec, args.workload, T),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


DECODE_T_MAX = 32   # largest T on the decode (GEMV) path; larger T takes the tcgen05 GEMMs


def launches_per_step(T: int, n_exp: int, ids_given: bool, f32: bool = False) -> int:
    """Kernels one colibri_moe_layer call launches. Decode (T <= 32): one kernel for q8 of
    x, router logits, selection (or the given ids), bucketing, gate/up, down and combine.
    Prefill: q8, router logits, selection, bucketing (q8 and bucketing alone with the ids
    given), the two tcgen05 GEMMs and the combine. The fp32-activation decode: router
    logits and selection (unless the ids are given), gate/up, down and the combine."""
    if f32:
        return 3 if ids_given else 5
    if T <= DECODE_T_MAX:
        return 1
    return 5 if ids_given else 7


def workload_config(spec, workload, T):
    return {"workload": workload, "d": spec.d, "ffn": spec.ffn, "n_exp": spec.n_exp, "top_k": spec.top_k,
            "shared_ffn": spec.shared_ffn if spec.has_shared else 0, "router": spec.router, "T": T,
            "experts_resident": "all in HBM",
            "l2": ("between timed steps a 256 MB buffer is written and another 256 MB buffer read, then "
                   "one call of the layer before (same shape, its own weights at other addresses): "
                   "code and small tables warm, none of this layer's weights, router or shared expert in L2"),
            "timing": "CUDA events per step around one CUDA-graph replay",
            "group": getattr(spec, "group", 32),
            "activations": "fp32" if is_f32(workload) else f"int8 (per-{getattr(spec, 'group', 32)}-group absmax)"}


# ---------------------------------------------------------------- expert streaming
STREAM_LAYERS = 8
STREAM_SLOTS = 512
LOOKAHEAD_ACCURACY = 0.716   # next-layer routing predictability stated by the pages


def stream_ops(ids_np, guess, predictor: str, n_exp: int, steps: int):
    """The cache operations of the streaming run, as colibri_lru_trace ops: per step and
    layer a lookup batch (kind 0, then kind 1 per id) and the next layer's prefetch
    (kind 2). Returns kinds, keys and the step of each op."""
    L_ = ids_np.shape[1]
    kinds, keys, step = [], [], []
    for s in range(steps):
        for l in range(L_):
            kinds.append(0); keys.append(0); step.append(s)
            for e in ids_np[s, l]:
                kinds.append(1); keys.append(l * n_exp + int(e)); step.append(s)
            nl, ns = (l + 1, s) if l + 1 < L_ else (0, s + 1)
            if predictor == "lookahead":
                pre = np.unique(guess[ns, nl])
            elif ns - 1 >= 0:
                pre = ids_np[ns - 1, nl]
            else:
                pre = []
            for e in pre:
                kinds.append(2); keys.append(nl * n_exp + int(e)); step.append(s)
    return np.array(kinds, np.int32), np.array(keys, np.int64), np.array(step)


def run_cache_sim(args):
    """Hit rates of the expert cache's policy on the streaming workload's ids, for several
    hot-set sizes, through the library's host-only trace of the policy."""
    from routed_expert_ffn_grouped_b300 import colibri as C
    spec, L_ = synth.GLM52, STREAM_LAYERS
    K, W = args.steps, args.warmup
    ids_np, _ = synth.streaming_ids(spec, args.seed, L_, W + K + 1)
    prng = np.random.default_rng([args.seed, 99])
    guess = ids_np.copy()
    wrong = prng.random(ids_np.shape) >= LOOKAHEAD_ACCURACY
    guess[wrong] = prng.integers(0, spec.n_exp, int(wrong.sum()))
    kinds, keys, step = stream_ops(ids_np, guess, args.predictor, spec.n_exp, W + K)
    timed = (kinds == 1) & (step >= W)
    rates = {}
    for n_hot in (0, 64, 128, 256, 384, STREAM_SLOTS - spec.top_k):
        res = C.colibri_lru_trace_hot(STREAM_SLOTS, n_hot, kinds, keys)
        rates[str(n_hot)] = float((res[timed] == 1).mean())
    line = {"metric": "expert cache hit rate (host simulation of the policy)", "unit": "fraction",
            "higher_is_better": True, "data": "synthetic",
            "config": {"workload": args.workload, "layers": L_, "n_exp": spec.n_exp, "top_k": spec.top_k,
                       "hbm_slots": STREAM_SLOTS, "hot_slots": args.hot_slots, "reuse": 0.7, "steps": K, "warmup": W,
                       "predictor": args.predictor},
            "hit_rate_by_hot_slots": rates}
    print(json.dumps(line), flush=True)


def interval_union(iv) -> float:
    """Total length of the union of intervals [a, b)."""
    tot, end = 0.0, float("-inf")
    for a, b in sorted(iv):
        if b <= end:
            continue
        tot += b - max(a, end)
        end = b
    return tot


def overlap_stats(copy_iv, compute_iv, window: float) -> dict:
    """Busy fractions of a window from the copy and compute intervals, and the share of
    copy time that ran beside compute (|A and B| = |A| + |B| - |A or B|)."""
    cu, pu = interval_union(copy_iv), interval_union(compute_iv)
    au = interval_union(list(copy_iv) + list(compute_iv))
    both = cu + pu - au
    return {"copy_busy_frac": cu / window, "compute_busy_frac": pu / window,
            "overlap_frac_of_copy": both / cu if cu > 0 else None, "idle_frac": 1.0 - au / window}


def h2d_peak_gbs(torch, src, dst, reps: int = 4) -> float:
    """Pinned host -> HBM copy rate of one large cudaMemcpyAsync, timed with CUDA events
    on its own stream (src pinned, dst on the device, both flat uint8)."""
    n = min(src.numel(), dst.numel())
    s = torch.cuda.Stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        dst[:n].copy_(src[:n], non_blocking=True)
        e0.record(s)
        for _ in range(reps):
            dst[:n].copy_(src[:n], non_blocking=True)
        e1.record(s)
    s.synchronize()
    return n * reps / (e0.elapsed_time(e1) / 1e3) / 1e9


def run_stream(args):
    """Decode T=1 through a stack of GLM-5.2-shaped layers whose routed experts live in
    pinned host memory (2048 blobs, ~48 GB) behind an HBM LRU cache of 512 slots
    (~12 GB); routing keeps each id from the previous step with probability 0.7. A layer's
    ids reach the host only once the previous layer has finished (the host waits on the
    compute stream, as a host-side cache must), unless --ids-ahead. Before each layer the
    next layer's experts are prefetched as predicted (previous step's ids, or an emulated
    router lookahead), as a queue of chunks that the host enqueues while it waits and that
    the next lookup finishes or cancels. The shared experts stay resident. A step is one
    token through all layers; the timed region includes the host's cache decisions. An
    instrumented pass after the timed one records CUDA events on the demand copy stream,
    the prefetch stream and the compute stream for the overlap figures."""
    import ctypes
    import torch
    from routed_expert_ffn_grouped_b300 import build as cbuild
    from routed_expert_ffn_grouped_b300 import colibri as C

    world, rank, local = dist_setup(torch)
    if rank == 0 or not os.path.exists(C.LIB_PATH):
        cbuild.build()
    barrier(torch, world)
    spec, T, L_ = synth.GLM52, 1, STREAM_LAYERS
    E = spec.n_exp
    K, W = args.steps, args.warmup
    nb = synth.blob_layout(spec.d, spec.ffn).nbytes
    t_gen = time.perf_counter()
    pinned = torch.empty((L_ * E, nb), dtype=torch.uint8, pin_memory=True)
    pn = pinned.numpy()
    # layer 0's experts are drawn; the other layers hold copies (content does not change
    # what is streamed or timed)
    for e in range(E):
        synth.fill_expert_blob(pn[e], spec.d, spec.ffn, args.seed, 0, e)
    for l in range(1, L_):
        pn[l * E:(l + 1) * E] = pn[:E]
    gen_s = time.perf_counter() - t_gen
    shared_blob = torch.from_numpy(synth.expert_blob(spec, args.seed, 0, 0, shared=True))
    shared_dev = [shared_blob.cuda() for _ in range(L_)]
    sl = C.colibri_blob_layout_for(spec.d, spec.shared_ffn)
    shared = [C.Expert(b.data_ptr() + sl.w1, b.data_ptr() + sl.w3, b.data_ptr() + sl.w2,
                       b.data_ptr() + sl.s1, b.data_ptr() + sl.s3, b.data_ptr() + sl.s2) for b in shared_dev]
    tables = (L_ * E * ctypes.sizeof(C.Expert) + 255) // 256 * 256
    pool = torch.empty(tables + STREAM_SLOTS * nb, dtype=torch.uint8, device="cuda")
    peak_n = min(2 << 30, STREAM_SLOTS * nb)
    h2d_peak = h2d_peak_gbs(torch, pinned.view(-1)[:peak_n], pool[tables:tables + peak_n])
    copy = torch.cuda.Stream()
    pcopy = torch.cuda.Stream()
    stream = torch.cuda.Stream()
    cache = C.ExpertCache(pool, pinned, L_, E, spec.d, spec.ffn, spec.top_k, copy)
    chunk = int(args.prefetch_chunk_mb * (1 << 20)) // 256 * 256
    cache.set_prefetch(pcopy, args.prefetch_inflight, chunk)
    if args.hot_slots:
        cache.set_hot(args.hot_slots)
    K2 = min(K, 24)                                 # instrumented steps after the timed ones
    ids_np, w_np = synth.streaming_ids(spec, args.seed, L_, W + K + K2 + 1)
    # emulated router lookahead: each id of the next layer is named correctly with the
    # pages' stated predictability (71.6%), else replaced by a popular-looking wrong id
    prng = np.random.default_rng([args.seed, 99])
    guess = ids_np.copy()
    wrong = prng.random(ids_np.shape) >= LOOKAHEAD_ACCURACY
    guess[wrong] = prng.integers(0, E, int(wrong.sum()))
    ids = torch.from_numpy(ids_np).cuda()          # [steps][layer][k]
    w = torch.from_numpy(w_np).cuda()
    cfg = C.layer_cfg(spec)
    xs = torch.from_numpy(np.stack([synth.activations(spec, args.seed, T, step=i) for i in range(16)])).cuda()
    out = torch.empty((T, spec.d), dtype=torch.float32, device="cuda")
    ws = torch.empty(C.colibri_moe_workspace_bytes(cfg, T), dtype=torch.uint8, device="cuda")

    def ev(q):
        e = torch.cuda.Event(enable_timing=True)
        e.record(q)
        return e

    def step(s, rec=None):
        for l in range(L_):
            if not args.ids_ahead:
                # layer l's ids exist once layer l-1 has run; prefetch chunks go out meanwhile
                p0 = ev(pcopy) if rec is not None else None
                cache.wait(stream, 60000)
                if rec is not None:
                    rec["copy"].append((p0, ev(pcopy)))
            d0 = ev(copy) if rec is not None else None
            cache.lookup(l, ids_np[s, l], wait_on=stream)
            if rec is not None:
                rec["copy"].append((d0, ev(copy)))
            nl, ns = (l + 1, s) if l + 1 < L_ else (0, s + 1)
            s0 = ev(pcopy) if rec is not None else None
            if args.predictor == "lookahead":
                cache.stage(nl, np.unique(guess[ns, nl]))   # next-layer prefetch, predicted
            elif ns - 1 >= 0:
                cache.stage(nl, ids_np[ns - 1, nl])         # the previous step's ids
            if rec is not None:
                rec["copy"].append((s0, ev(pcopy)))         # whole-blob prefetches, if any
            c0 = ev(stream) if rec is not None else None
            C.colibri_moe_layer(cfg, xs[(s * L_ + l) % 16], None, None, cache.table(l), shared[l],
                                ids[s, l].view(1, -1), w[s, l].view(1, -1), True, out, ws, stream=stream)
            if rec is not None:
                rec["compute"].append((c0, ev(stream)))

    for s in range(W):
        step(s)
    stream.synchronize()
    cache.sync(60000)
    st0 = cache.stats()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(torch, world)
    torch.cuda.synchronize()
    sampler = ClockSampler(torch, local)
    t0 = time.perf_counter()
    with sampler:
        ev0.record(stream)
        for s in range(W, W + K):
            step(s)
        ev1.record(stream)
        torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ms = allreduce_max(torch, world, ev0.elapsed_time(ev1))
    st1 = cache.stats()
    d = {k: st1[k] - st0[k] for k in st1 if k != "n_slots"}
    value = world * T * K / (ms / 1e3)
    # instrumented pass: events on the three streams (not part of the timed value)
    rec = {"copy": [], "compute": []}
    cache.sync(60000)
    torch.cuda.synchronize()
    base = ev(stream)
    for s in range(W + K, W + K + K2):
        step(s, rec)
    end = ev(stream)
    torch.cuda.synchronize()
    cache.sync(60000)
    rel = lambda pairs: [(base.elapsed_time(a), base.elapsed_time(b)) for a, b in pairs]
    overlap = overlap_stats(rel(rec["copy"]), rel(rec["compute"]), base.elapsed_time(end))
    overlap["steps"] = K2
    overlap["how"] = ("CUDA events on the demand copy stream around each lookup, on the prefetch stream "
                      "around each host wait and each prefetch call, on the compute stream around each "
                      "layer call")
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "i8xi4->i32, f32", "data": "synthetic",
            "config": {"workload": args.workload, "layers": L_, "d": spec.d, "ffn": spec.ffn, "n_exp": E,
                       "top_k": spec.top_k, "T": T, "host_blobs": L_ * E, "host_bytes": L_ * E * nb,
                       "hbm_slots": STREAM_SLOTS, "hot_slots": args.hot_slots, "reuse": 0.7,
                       "prefetch": ("next layer's ids from an emulated lookahead, 71.6% correct"
                                    if args.predictor == "lookahead" else "previous step's ids of the next layer"),
                       "prefetch_chunk_bytes": chunk, "prefetch_inflight": args.prefetch_inflight,
                       "host_waits_for_previous_layer": not args.ids_ahead,
                       "timing": "CUDA events around K steps on the compute stream; host cache decisions inside"},
            "cache": {"hit_rate": d["hits"] / max(1, d["lookups"]), "lookups": d["lookups"],
                      "misses": d["misses"], "prefetch_staged": d["prefetch_staged"],
                      "prefetch_used": d["prefetch_used"], "prefetch_cancelled": d["prefetch_cancelled"],
                      "prefetch_accuracy": d["prefetch_used"] / max(1, d["prefetch_staged"]),
                      "bytes_staged": d["bytes_staged"], "prefetch_bytes": d["prefetch_bytes"],
                      "pcie_gbs": d["bytes_staged"] / (ms / 1e3) / 1e9,
                      "h2d_peak_gbs": h2d_peak,
                      "staging_frac_of_peak": d["bytes_staged"] / (ms / 1e3) / 1e9 / h2d_peak},
            "overlap": overlap,
            "wall_s": wall, "generate_s": gen_s,
            # one per layer call (ids given) + one table-entry write per blob staged to the end
            "gpu_launches": K * L_ * launches_per_step(T, E, True) + d["misses"]
                            + d["prefetch_staged"] - d["prefetch_cancelled"],
            "clocks": sampler.summary(),
        }
        print(json.dumps(line), flush=True)
    cache.close()


# ---------------------------------------------------------------- GPU arm
def run_colibri(args):
    import torch
    from routed_expert_ffn_grouped_b300 import build as cbuild
    from routed_expert_ffn_grouped_b300 import colibri as C

    world, rank, local = dist_setup(torch)
    if rank == 0 or not os.path.exists(C.LIB_PATH):
        cbuild.build()
    barrier(torch, world)
    name, T, row_scale = WORKLOADS[args.workload]
    spec = synth.SPECS[name]
    host = synth.make_layer(spec, args.seed)
    dl = C.DeviceLayer(host)
    stream = torch.cuda.Stream()
    xs_host = np.stack([synth.activations(spec, args.seed, T, step=i, row_scale=row_scale) for i in range(N_X)])
    xs = torch.from_numpy(xs_host).cuda()
    x = torch.empty((T, spec.d), dtype=torch.float32, device="cuda")
    out = torch.empty((T, spec.d), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda")
    f32 = is_f32(args.workload)
    layer_fn = C.colibri_moe_layer_f32 if f32 else C.colibri_moe_layer
    ws_bytes = (C.colibri_moe_f32_workspace_bytes if f32 else C.colibri_moe_workspace_bytes)(dl.cfg, T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    scrub = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    # the layer before: same shape, its own weights (as in a model, where the previous
    # layer's call leaves code and small tables warm but none of this layer's data)
    prev = C.DeviceLayer.twin(dl, shift=spec.n_exp // 3)
    x_prev = torch.from_numpy(synth.activations(spec, args.seed + 1, T, row_scale=row_scale)).cuda()
    out_prev = torch.empty_like(out)
    ids_prev, w_prev = torch.empty_like(ids), torch.empty_like(w)
    ws_prev = torch.empty_like(ws)
    K, W = args.steps, args.warmup
    ids_log = torch.empty((W + K, T, spec.top_k), dtype=torch.int32, device="cuda")

    def layer():
        layer_fn(dl.cfg, x, dl.Wr, dl.bias, dl.table, dl.shared, ids, w, False, out, ws,
                 stream=torch.cuda.current_stream())

    with torch.cuda.stream(stream):
        x.copy_(xs[0])
        layer()                                   # eager warm call (also checks the status)
        stream.synchronize()
        st = C.colibri_workspace_status(dl.cfg, T, ws, stream=stream)
        if st != C.OK:
            raise RuntimeError(f"layer reported device error {st}")
    def layer_prev():
        layer_fn(prev.cfg, x_prev, prev.Wr, prev.bias, prev.table, prev.shared, ids_prev, w_prev, False,
                 out_prev, ws_prev, stream=torch.cuda.current_stream())

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        layer()
    graph_prev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_prev, stream=stream):
        layer_prev()
    C.colibri_moe_profile_enable(True)
    graph_prof = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_prof, stream=stream):
        layer()
    C.colibri_moe_profile_enable(False)

    def pre(i):
        x.copy_(xs[i % N_X])
        flush.fill_(float(i))
        scrub.sum()
        graph_prev.replay()

    # warm-up
    with torch.cuda.stream(stream):
        for i in range(W):
            pre(i)
            graph.replay()
            ids_log[i].copy_(ids)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    barrier(torch, world)
    torch.cuda.synchronize()
    sampler = ClockSampler(torch, local)
    with sampler, torch.cuda.stream(stream):
        for i in range(K):
            pre(W + i)
            starts[i].record(stream)
            graph.replay()
            ends[i].record(stream)
            ids_log[W + i].copy_(ids)
        torch.cuda.synchronize()
    barrier(torch, world)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = allreduce_max(torch, world, float(sum(step_ms)))
    value = weak_scaling_value(world, T, K, total_ms)

    # informational: the same replays without the L2 flush between them (what back-to-back
    # layers of a model see: weights still stream from HBM, code and small tables stay warm)
    KB = min(K, 1000)
    nf_s = [torch.cuda.Event(enable_timing=True) for _ in range(KB)]
    nf_e = [torch.cuda.Event(enable_timing=True) for _ in range(KB)]
    with torch.cuda.stream(stream):
        for i in range(KB):
            x.copy_(xs[(W + i) % N_X])
            nf_s[i].record(stream)
            graph.replay()
            nf_e[i].record(stream)
        torch.cuda.synchronize()
    nf_ms = float(np.mean([a.elapsed_time(b) for a, b in zip(nf_s, nf_e)]))

    # expert bytes per step: distinct routed experts + the shared expert
    nb, gu_b, dn_b = blob_bytes(spec, spec.ffn)
    sh = blob_bytes(spec, spec.shared_ffn) if spec.has_shared else (0, 0, 0)
    ids_np = ids_log[W:].cpu().numpy()
    distinct = np.array([len(np.unique(ids_np[i])) for i in range(K)])
    expert_bytes = distinct * nb + sh[0]
    gu_bytes = distinct * gu_b + sh[1]
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    layer_gbs = float(np.sum(expert_bytes) / (sum(step_ms) / 1e3) / 1e9)

    # per-kernel profiling pass (events between the kernels, recorded inside the graph)
    P = min(K, 400)
    prof = {k: [] for k in C.PROFILE_KERNELS}
    prof_bytes = []
    prefill = T > DECODE_T_MAX
    with torch.cuda.stream(stream):
        for i in range(P):
            pre(W + i)
            graph_prof.replay()
            ms = C.colibri_moe_profile_read()
            for k, v in ms.items():
                prof[k].append(v)
            u = len(np.unique(ids.cpu().numpy()))
            # algorithmic bytes of the roofline kernel: gate/up weights for the prefill
            # GEMM, all expert weights for the fused decode kernel
            prof_bytes.append(u * gu_b + sh[1] if prefill else u * nb + sh[0])
    mean = {k: float(np.mean(v)) for k, v in prof.items()}
    if f32:
        kern_ms = {"k_route_logits": mean["router_logits"], "k_router_select": mean["router_select"],
                   "k_f32_gateup": mean["gateup"], "k_f32_down": mean["down"], "k_combine": mean["combine"],
                   "event_records": mean["q8"] + mean["bucket"]}
        roof_ms = np.array(prof["gateup"]) + np.array(prof["down"])
        gu_kernel = "k_f32_gateup + k_f32_down (fp32 activations; weights read once per pair)"
        traffic = None
    elif prefill:
        kern_ms = {"k_q8 + k_route_logits_tiled": mean["router_logits"], "k_router_select": mean["router_select"],
                   "k_bucket": mean["bucket"], "k_gemm<0>": mean["gateup"], "k_gemm<1>": mean["down"],
                   "k_combine": mean["combine"]}
        roof_ms = np.array(prof["gateup"])
        gu_kernel = "k_gemm<0> (tcgen05 gate/up + SwiGLU + q8)"
        traffic = None
    else:
        # one kernel; the other slots hold only the time of an event record
        kern_ms = {"k_decode": mean["gateup"],
                   "event_records": mean["q8"] + mean["router_logits"] + mean["router_select"] + mean["bucket"]
                   + mean["down"] + mean["combine"]}
        roof_ms = np.array(prof["gateup"])
        gu_kernel = "k_decode (q8 of x, router logits, selection, bucketing, gate/up, down, combine)"
        traffic = traffic_from_profiles("k_decode_glm52_decode_t1", "kernels_decode.cu", args.workload)
    gu_gbs = float(np.mean(np.array(prof_bytes) / (roof_ms / 1e3)) / 1e9)
    roof_tensor = None
    if prefill:
        # the same kernel against the tensor peak: algorithmic MACs of gate/up, routed
        # pairs and the shared expert, x 2 flops
        flops = 2.0 * T * spec.d * 2 * (spec.top_k * spec.ffn + (spec.shared_ffn if spec.has_shared else 0))
        tf = flops / (float(np.mean(prof["gateup"])) / 1e3) / 1e12
        tpeak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
        roof_tensor = {"bound": "tensor", "kernel": gu_kernel, "achieved": tf, "peak": tpeak, "unit": "TFLOP/s",
                       "frac": tf / tpeak, "algorithmic_flops_per_launch": flops,
                       "peak_source": f"MEASURED_PEAKS.json bf16_tflops ({peak_kind})"}

    # end to end through the public API: one blocking colibri_moe_layer_host call per step,
    # x from pinned host memory in, out (and the device error flag) back to pinned host
    x_pin = torch.from_numpy(xs_host).pin_memory()
    out_pin = torch.empty((T, spec.d), dtype=torch.float32).pin_memory()
    ws_host = None if f32 else torch.empty(C.colibri_moe_host_workspace_bytes(dl.cfg, T), dtype=torch.uint8,
                                           device="cuda")
    # at least 200 timed calls (whatever --steps is) after 50 warm-up calls: a host-side
    # figure needs more samples than the device-timed steps to be stable
    KE = min(max(K, 200), 500)
    e2e_s = 0.0

    def e2e_call(i):
        if f32:
            x.copy_(x_pin[i % N_X], non_blocking=True)
            layer_fn(dl.cfg, x, dl.Wr, dl.bias, dl.table, dl.shared, ids, w, False, out, ws, stream=stream)
            out_pin.copy_(out, non_blocking=True)
            stream.synchronize()
        else:
            C.colibri_moe_layer_host(dl.cfg, x_pin[i % N_X], dl.Wr, dl.bias, dl.table, dl.shared, None, None,
                                     False, out_pin, ws_host, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(max(W, 50)):              # untimed warm-up calls of the same entry point
            e2e_call(i)
        stream.synchronize()
        for i in range(KE):
            flush.fill_(float(i))
            scrub.sum()
            graph_prev.replay()
            stream.synchronize()
            t0 = time.perf_counter()
            e2e_call(i)
            e2e_s += time.perf_counter() - t0
    e2e_s = allreduce_max(torch, world, e2e_s)
    e2e_value = world * T * KE / e2e_s

    cpu = None
    cpu_all = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # batches of at most 8 of the workload's tokens: the oracle's work per token does
        # not depend on the batch, and a 2048-token batch would run for minutes
        tb = min(T, 8)
        rate, n, dt = oracle_tokens_per_s(spec, host, [xs_host[i][:tb] for i in range(N_X)], 15.0, 64,
                                          act="f32" if f32 else "q8")
        cpu = {"value": rate * tb, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} batches of {tb} tokens of {args.workload} through the C oracle "
                         f"({dt:.1f} s, single-threaded)"}
        if prefill:
            # prefill is minutes of oracle work per batch single-threaded: also the oracle
            # on every host core (informational, beside the single-core baseline)
            rate_a, n_a, dt_a, thr = oracle_tokens_per_s_all_cores(
                spec, host, [xs_host[i][:1] for i in range(N_X)], 15.0, act="f32" if f32 else "q8")
            cpu_all = {"value": rate_a, "unit": "tokens/s", "cores": thr, "kind": "oracle",
                       "sample": f"{n_a} tokens of {args.workload}, one token per oracle call, {thr} host "
                                 f"threads ({dt_a:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("i4 x f32 -> f32" if f32 else "bf16xbf16->f32 (int4 and q8 codes, exact in bf16)" if prefill
                      else "i8xi4->i32, f32"),
            "data": "synthetic",
            "config": workload_config(spec, args.workload, T),
            "expert_hbm_gbs": layer_gbs, "expert_hbm_frac": layer_gbs / hbm_peak,
            "expert_bytes_per_step": float(np.mean(expert_bytes)),
            "roofline": {"bound": "hbm", "kernel": gu_kernel, "achieved": gu_gbs, "peak": hbm_peak,
                         "unit": "GB/s", "frac": gu_gbs / hbm_peak, "traffic": traffic,
                         "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})",
                         "algorithmic_bytes_per_launch": float(np.mean(prof_bytes))},
            "roofline_tensor": roof_tensor,
            "kernel_ms": kern_ms,
            "no_l2_flush": {"value": world * T / (nf_ms / 1e3), "ms_per_step": nf_ms, "steps": KB,
                            "note": "informational; the headline value flushes L2 between steps"},
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": T * spec.d * 4,
                    "d2h_bytes_per_step": T * spec.d * 4 + (0 if f32 else 4), "steps": KE,
                    "path": ("colibri_moe_layer_f32 between pinned-host copies of x and out, eager launches"
                             if f32 else "colibri_moe_layer_host (pinned host x and out, the error flag read "
                             "back) via the Python binding, eager launches")},
            "gpu_launches": launches_per_step(T, spec.n_exp, False, f32) * K,
            "expert_load": informational(expert_load, ids_np, spec.n_exp),
            "host": informational(host_info),
            "clocks": sampler.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_stack_decode(args):
    """Eight resident layers of one shape per step, each with activations of its own (as when
    attention sits between a model's MoE layers; a bare chain of SwiGLU layers, out into x,
    overflows within a few layers): one colibri_moe_stack_decode launch, timed with CUDA
    events around a graph replay, beside the same eight layers as eight colibri_moe_layer
    calls in one graph. The layers are one drawn layer and device copies of it whose
    router rows are rolled (each routes elsewhere, and their weights sit at other
    addresses); 8 x 6 GB of GLM-shaped weights keep every step's bytes far above the L2
    (the OLMoE-shaped stack, 8 x 0.25 GB, streams its 8 x 31.5 MB per step through it)."""
    import torch
    from routed_expert_ffn_grouped_b300 import build as cbuild
    from routed_expert_ffn_grouped_b300 import colibri as C

    world, rank, local = dist_setup(torch)
    if rank == 0 or not os.path.exists(C.LIB_PATH):
        cbuild.build()
    barrier(torch, world)
    name, T, _ = WORKLOADS[args.workload]
    spec = synth.SPECS[name]
    L_ = STACK_LAYERS
    base = C.DeviceLayer(synth.make_layer(spec, args.seed))
    layers = [base] + [C.DeviceLayer.twin(base, shift=(spec.n_exp // L_) * l + 1) for l in range(1, L_)]
    stream = torch.cuda.Stream()
    xs = torch.from_numpy(np.stack([synth.activations(spec, args.seed, T, step=i) for i in range(N_X)])).cuda()
    xl = [torch.empty((T, spec.d), dtype=torch.float32, device="cuda") for _ in range(L_)]
    x = xl[0]
    outs = [torch.empty((T, spec.d), dtype=torch.float32, device="cuda") for _ in range(L_)]
    ids = [torch.empty((T, spec.top_k), dtype=torch.int32, device="cuda") for _ in range(L_)]
    w = [torch.empty((T, spec.top_k), dtype=torch.float32, device="cuda") for _ in range(L_)]
    cfg = base.cfg
    ws_stack = torch.empty(C.colibri_moe_stack_workspace_bytes(cfg, T), dtype=torch.uint8, device="cuda")
    ws = torch.empty(C.colibri_moe_workspace_bytes(cfg, T), dtype=torch.uint8, device="cuda")
    st = [dict(x=xl[l], Wr=dl.Wr, bias=dl.bias, experts=dl.table, shared=dl.shared, ids=ids[l], w=w[l],
               out=outs[l]) for l, dl in enumerate(layers)]

    def stacked():
        C.colibri_moe_stack_decode(cfg, x, st, False, ws_stack, stream=torch.cuda.current_stream())

    def sequential():
        for l, dl in enumerate(layers):
            C.colibri_moe_layer(cfg, xl[l], dl.Wr, dl.bias, dl.table, dl.shared, ids[l], w[l], False, outs[l], ws,
                                stream=torch.cuda.current_stream())

    def fill(i):
        for l in range(L_):
            xl[l].copy_(xs[(i + l) % N_X])

    with torch.cuda.stream(stream):
        fill(0)
        stacked()
        stream.synchronize()
        if C.colibri_workspace_status(cfg, T, ws_stack, stream=stream) != C.OK:
            raise RuntimeError("layer stack reported a device error")
    graphs = {}
    for key, fn in (("stack", stacked), ("sequential", sequential)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        graphs[key] = g
    K, W = args.steps, args.warmup
    ids_log = torch.empty((K, L_, T, spec.top_k), dtype=torch.int32, device="cuda")

    def timed(g, log):
        with torch.cuda.stream(stream):
            for i in range(W):
                fill(i)
                g.replay()
        torch.cuda.synchronize()
        s_ev = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        with torch.cuda.stream(stream):
            for i in range(K):
                fill(W + i)
                s_ev[i].record(stream)
                g.replay()
                e_ev[i].record(stream)
                if log:
                    for l in range(L_):
                        ids_log[i, l].copy_(ids[l])
            torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in zip(s_ev, e_ev)]

    barrier(torch, world)
    sampler = ClockSampler(torch, local)
    with sampler:
        step_ms = timed(graphs["stack"], True)
    total_ms = allreduce_max(torch, world, float(sum(step_ms)))
    seq_ms = timed(graphs["sequential"], False)
    if (C.colibri_workspace_status(cfg, T, ws_stack, stream=stream) != C.OK or
            C.colibri_workspace_status(cfg, T, ws, stream=stream) != C.OK):
        raise RuntimeError("a layer reported a device error")
    value = weak_scaling_value(world, T * L_, K, total_ms)
    nb, _, _ = blob_bytes(spec, spec.ffn)
    sh = blob_bytes(spec, spec.shared_ffn)[0] if spec.has_shared else 0
    ids_np = ids_log.cpu().numpy()
    step_bytes = np.array([sum(len(np.unique(ids_np[i, l])) * nb + sh for l in range(L_)) for i in range(K)])
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    achieved = float(np.sum(step_bytes) / (sum(step_ms) / 1e3) / 1e9)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s (layer-tokens: tokens x layers)",
            "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": total_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "i8xi4->i32, f32", "data": "synthetic",
            "config": dict(workload_config(spec, args.workload, T), layers=L_, inputs="each layer its own activations (no chaining)",
                           l2="no flush between steps: each step reads 8 layers' weights once",
                           timing="CUDA events per step around one CUDA-graph replay of the 8-layer launch"),
            "us_per_layer": total_ms / K / L_ * 1e3,
            "sequential_us_per_layer": float(np.mean(seq_ms)) / L_ * 1e3,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": None,
                         "kernel": "k_decode_stack (all 8 layers)",
                         "bytes": "per layer: distinct routed experts x blob bytes + the shared expert",
                         "peak_kind": peak_kind},
            "gpu_launches": K,
            "e2e": None,
            "cpu_baseline": None,
            "clocks": sampler.summary(),
        }
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "glm52_stream_8l":
        run_cache_sim(args) if args.cache_sim else run_stream(args)
    elif args.workload.endswith("_stack8"):
        run_stack_decode(args)
    else:
        run_colibri(args)


if __name__ == "__main__":
    main()
