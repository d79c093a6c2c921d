"""The multi-rank side of bench.py at world size 2, on CPU with gloo.

Each rank runs its own replica on its own batch; the only cross-rank steps are
the barrier and the max of the step times. These tests run that logic in two
real processes (gloo, 127.0.0.1) without a GPU: the max is taken across ranks,
the whole-job value counts every rank's work over the slowest rank's time, the
per-rank batches differ, and a rank that drops out is seen by the other as an
error of the collective (host-side failure, bounded by the group's timeout).
"""
from __future__ import annotations

import datetime
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port, timeout_s=60):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=timeout_s))


def _worker_aggregate(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    from context_causal_attention_headtail_gb300.synth import WORKLOADS, make_inputs, make_workload
    _init(rank, world, port)
    w_env, r_env, l_env = bench.rank_env()
    assert (w_env, r_env, l_env) == (world, rank, rank)
    dist.barrier()
    ms_local = 10.0 + 5.0 * rank                       # rank 1 is the slower one
    ms = bench.max_over_ranks(ms_local, world, device="cpu")
    w = WORKLOADS["window_32k"]
    value = bench.weak_scaling_value(world, w.fwdbwd_flops(), ms)
    small = make_workload("rank_batch", B=1, T=64, H=1, d=64, cp=2)
    x = make_inputs(small, bench.rank_seed(small, rank))["q"].float()
    xs = [torch.zeros_like(x) for _ in range(world)]
    dist.all_gather(xs, x)
    out[rank] = (ms, value, bool(torch.equal(xs[0], xs[1])))
    dist.destroy_process_group()


@pytest.mark.timeout(180)
def test_two_rank_timing_aggregation():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker_aggregate, args=(world, port, out), nprocs=world, start_method="spawn")
    from context_causal_attention_headtail_gb300.synth import WORKLOADS
    flops = WORKLOADS["window_32k"].fwdbwd_flops()
    for r in range(world):
        ms, value, same = out[r]
        assert ms == 15.0                              # the max over ranks, on every rank
        assert abs(value - 2 * flops / 15e-3 / 1e12) < 1e-9
        assert not same                                # each rank has its own batch


def _worker_dropout(rank, world, port, out):
    _init(rank, world, port, timeout_s=5)
    dist.barrier()
    if rank == 1:                                      # leaves between steps, nothing in flight
        os._exit(0)
    try:
        t = torch.ones(1)
        dist.all_reduce(t)
        out[rank] = "completed"
    except Exception as e:                             # gloo reports the lost peer or the timeout
        out[rank] = "error: " + type(e).__name__


@pytest.mark.timeout(180)
def test_rank_dropout_is_an_error_not_a_hang():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    ctx = mp.start_processes(_worker_dropout, args=(world, port, out), nprocs=world, start_method="spawn",
                             join=False)
    for p in ctx.processes:
        p.join(120)
    assert out.get(0, "").startswith("error"), out.get(0)


def test_launch_plan_honours_gpus():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.launch_plan(1, {}) == ("run", "")
    assert bench.launch_plan(4, {})[0] == "relaunch"
    assert bench.launch_plan(2, {"WORLD_SIZE": "2"}) == ("run", "")
    assert bench.launch_plan(8, {"WORLD_SIZE": "1"})[0] == "refuse"
    assert bench.launch_plan(0, {})[0] == "refuse"
    cmd = bench.relaunch_cmd(2, ["--gpus", "2", "--steps", "1"], 29999)
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=2" in cmd and cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[-4:] == ["--gpus", "2", "--steps", "1"]


def _bench(args, extra_env=None, timeout=300):
    import subprocess
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    env.update(extra_env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, env=env,
                          capture_output=True, text=True, timeout=timeout)


@pytest.mark.timeout(120)
def test_bench_refuses_a_world_size_other_than_gpus():
    r = _bench(["--gpus", "2", "--impl", "reference"], {"WORLD_SIZE": "1", "RANK": "0"})
    assert r.returncode == 2 and "WORLD_SIZE=1" in r.stderr
    assert r.stdout.strip() == ""


@pytest.mark.timeout(400)
def test_bench_gpus_2_starts_two_ranks():
    """--gpus 2 without a launcher starts two ranks (gloo-free: the oracle arm
    needs no collective); rank 0 alone prints, with n_gpus = 2."""
    import json
    r = _bench(["--gpus", "2", "--impl", "reference", "--workload", "tiny_fp32",
                "--steps", "1", "--warmup", "0"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2

