"""Multi-process host logic of the benchmark, on CPU with the gloo backend.

The hot path shards into independent replicas (no collective on the data
path); the only cross-rank step is the timing reduction: every rank reports
its own elapsed time and the job's time is the slowest rank's.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        local = [10.0 * (rank + 1), 1.0 + rank, 5.0 - rank]
        got = bench.reduce_max(dist, local, torch.device("cpu"))
        # replicas: every rank builds the same seeded workload independently
        from gqa_attention_head_sink_gb300 import workloads
        inp = workloads.make_prefill([40, 7], num_q_heads=4, num_kv_heads=2, seed=3)
        digest = torch.tensor([float(inp.q.float().sum()), float(inp.sinks.sum())], dtype=torch.float64)
        gathered = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(gathered, digest)
        q.put((rank, got, [g.tolist() for g in gathered]))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction_and_replicas():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, gathered in results:
        assert got == [20.0, 2.0, 5.0]  # slowest rank wins, element-wise
        assert gathered[0] == gathered[1]  # identical replicas


def test_reduce_max_without_process_group():
    import bench
    assert bench.reduce_max(None, [1.0, 2.0], torch.device("cpu")) == [1.0, 2.0]


def test_both_arms_report_the_same_workload():
    # the reference arm (the oracle on host cores) and the GPU arm name one config, so the two
    # lines compare the same metric on the same workload
    import bench
    for world in (1, 2, 8):
        cfg = bench._config(world)
        assert cfg == bench._config(world) and "seq 8192" in cfg["workload"] and "num_splits 8" in cfg["workload"]
    assert bench._config(1)["parallelism"] == "single GPU" and bench._config(4)["parallelism"] == "replicas x4"


def test_traffic_is_reported_only_for_the_captured_source():
    # the per-launch DRAM bytes come from the committed capture only while the kernel source is
    # the captured one: any other source hash reads as "not measured"
    import bench
    assert bench._traffic("no_such_kernel", bench.PREFILL_SOURCES) is None
    for line in open(os.path.join(bench.ROOT, "profiles", "dram_traffic.txt")):
        if line.startswith("#") or not line.strip():
            continue
        name, digest, nbytes = line.split()[:3]
        assert len(digest) == 16 and float(nbytes) > 0


def test_reference_arm_runs_the_requested_steps(monkeypatch):
    # the reference arm times exactly --steps / --warmup steps, each a sample sized from one
    # timed head and one timed sequence (fakes stand in for the float64 oracle here)
    import argparse
    import bench
    calls = {"pre": [], "dec": []}

    def fake_pre(pre, nh=bench.PREFILL_SAMPLE_HEADS):
        calls["pre"].append(nh)
        return 0.05 * nh, 1000 * nh

    def fake_dec(dec, seqs=8):
        calls["dec"].append(seqs)
        return 0.01 * seqs, 100 * seqs

    monkeypatch.setattr(bench, "_oracle_prefill_sample", fake_pre)
    monkeypatch.setattr(bench, "_oracle_decode_sample", fake_dec)
    monkeypatch.setattr(bench.workloads, "workload", lambda name, device="cpu": argparse.Namespace(num_q_heads=64))
    monkeypatch.setattr(bench.workloads, "make_decode", lambda *a, **k: argparse.Namespace(batch=16))
    for steps, warm in [(20, 3), (1000, 10), (1, 0)]:
        calls["pre"].clear()
        calls["dec"].clear()
        line = bench.run_reference(argparse.Namespace(steps=steps, warmup=warm), None, 0, 1)
        assert line["steps"] == steps and line["warmup"] == warm
        # one calibration call each, then warm-up + steps samples of one size
        assert calls["pre"][0] == 1 and calls["dec"][0] == 1
        nh, ns = calls["pre"][-1], calls["dec"][-1]
        assert len(calls["pre"]) == 1 + warm + steps and set(calls["pre"][1:]) == {nh}
        assert len(calls["dec"]) == 1 + warm + steps and set(calls["dec"][1:]) == {ns}
        assert nh & (nh - 1) == 0 and 1 <= nh <= 64 and 1 <= ns <= 16
        per_step = min(4.0, bench.REFERENCE_BUDGET_S / (steps + warm))
        assert nh == 1 or 0.05 * nh <= 0.85 * per_step
        assert line["value"] == round(1000 * nh * steps / (0.05 * nh * steps) / 1e12, 6)
    assert bench.run_reference(argparse.Namespace(steps=3, warmup=1), None, 1, 2) is None  # other ranks: no work
