"""The multi-rank harness of bench.py on CPU: two gloo ranks set up the process group from
the launcher's environment, meet at the barrier, agree on the slowest rank's time, and
report the whole-job (weak-scaling) throughput; the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import bench
    w, r, _ = bench.dist_setup(torch)
    bench.barrier(torch, w)
    my_ms = 10.0 + 5.0 * r                      # rank 1 is the slow one
    mx = bench.allreduce_max(torch, w, my_ms)
    val = bench.weak_scaling_value(w, 4, 20, mx)
    out.put((r, w, mx, val))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got.sort()
    assert [g[0] for g in got] == [0, 1] and all(g[1] == 2 for g in got)
    assert all(g[2] == pytest.approx(15.0) for g in got)          # max over ranks
    # 2 ranks x 4 tokens x 20 steps in the slowest rank's 15 ms
    assert all(g[3] == pytest.approx(2 * 4 * 20 / 0.015) for g in got)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.allreduce_max(None, 1, 3.5) == 3.5
    assert bench.weak_scaling_value(1, 1, 10, 1.0) == pytest.approx(10_000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    """Under torchrun the oracle arm is rank 0's alone: rank 1 returns at once (no output)."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    class Args:  # what run_reference would read after its rank check
        workload, steps, warmup, seed = "glm52_decode_t1", 1, 0, 0
    assert bench.run_reference(Args()) is None


def test_launch_counts_and_workload_tags():
    """The kernel launches the bench claims per layer call, by path, match the entry points'
    documented launch sequences; every workload names its activation type."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.launches_per_step(1, 256, False) == 1          # one kernel routes and runs the experts
    assert bench.launches_per_step(32, 256, False) == 1
    assert bench.launches_per_step(4, 256, True) == 1
    assert bench.launches_per_step(2048, 256, False) == 7
    assert bench.launches_per_step(2048, 256, True) == 5
    assert bench.launches_per_step(1, 256, False, f32=True) == 5   # logits, select, gate/up, down, combine
    assert bench.launches_per_step(1, 256, True, f32=True) == 3
    for name in bench.WORKLOADS:
        spec_name, T, _ = bench.WORKLOADS[name]
        from routed_expert_ffn_grouped_b300 import synth
        cfg = bench.workload_config(synth.SPECS[spec_name], name, T)
        assert cfg["workload"] == name
        gq = 64 if name.endswith("_g64") else 32
        assert cfg["group"] == gq
        assert cfg["activations"] == ("fp32" if name.endswith("_f32") else f"int8 (per-{gq}-group absmax)")
        if name.endswith("_f32"):
            assert T <= bench.DECODE_T_MAX     # the fp32-activation variant is decode only


def test_expert_load_and_host_fields():
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    # two steps of 2 tokens x top-2 over 4 experts
    ids = np.array([[[0, 1], [0, 2]],
                    [[3, 3], [3, 3]]], np.int32)
    ld = bench.expert_load(ids, 4)
    assert ld["steps"] == 2 and ld["pairs_per_step"] == 4.0
    assert ld["distinct_experts"] == (3 + 1) / 2
    assert ld["max_tokens_per_expert"] == (2 + 4) / 2
    assert ld["max_over_mean"] == (2 / 1 + 4 / 1) / 2           # mean per expert = 4 pairs / 4
    assert ld["tokens_per_expert_p50_p90_p99"][0] == float(np.percentile([2, 1, 1, 0, 0, 0, 0, 4], 50))
    h = bench.host_info()
    assert h["nproc"] and h["nproc"] >= 1
    assert bench.informational(lambda: 1 / 0)["error"].startswith("ZeroDivisionError")


def test_interval_overlap_arithmetic():
    """The streaming overlap figures: union lengths and the copy time that ran beside
    compute, on hand-made intervals."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.interval_union([]) == 0.0
    assert bench.interval_union([(0, 2), (1, 3), (5, 6)]) == 4.0
    assert bench.interval_union([(0, 10), (2, 3)]) == 10.0
    o = bench.overlap_stats([(0, 4), (6, 8)], [(3, 7)], 10.0)
    assert o["copy_busy_frac"] == pytest.approx(0.6)
    assert o["compute_busy_frac"] == pytest.approx(0.4)
    assert o["overlap_frac_of_copy"] == pytest.approx(2 / 6)      # [3,4) and [6,7)
    assert o["idle_frac"] == pytest.approx(0.2)                   # [8,10)
    assert bench.overlap_stats([], [(0, 1)], 2.0)["overlap_frac_of_copy"] is None
