"""The multi-GPU path is replicas only (no cross-GPU exchange). Its host-side
logic -- the max-over-ranks reduction and the whole-job time per call -- is
checked here with two gloo ranks on the CPU."""
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


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    per_rank_total_us = [1000.0, 1500.0][rank]
    worst = bench.reduce_max(per_rank_total_us, world)
    value = bench.aggregate_us_per_call(worst, steps=10, world=world)
    bench.barrier(world)
    q.put((rank, worst, value))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst, value in results:
        assert worst == 1500.0            # max over ranks
        assert value == 1500.0 / (10 * 2)  # whole-job time per call over both replicas


def test_single_rank_helpers():
    import bench
    assert bench.reduce_max(3.0, 1) == 3.0
    assert bench.aggregate_us_per_call(200.0, 4, 1) == 50.0


def _bench_cmd(*args):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    return [sys.executable, os.path.join(root, "bench.py"), *args]


def test_gpus_flag_starts_replica_ranks():
    """`bench.py --gpus 2` outside torchrun starts two ranks itself (gloo on
    the CPU); rank 0 alone prints the line, which reports both GPUs."""
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run(_bench_cmd("--gpus", "2", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                                  "--warmup", "0", "--ref-budget", "0.2"),
                       capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    assert lines[0]["n_gpus"] == 2 and lines[0]["impl"] == "reference"


def test_gpus_flag_must_match_world_size():
    import subprocess
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    r = subprocess.run(_bench_cmd("--gpus", "1", "--impl", "reference", "--workload", "tiny", "--steps", "1"),
                       capture_output=True, text=True, timeout=120, env=env)
    assert r.returncode != 0
    assert "WORLD_SIZE=2" in r.stderr
