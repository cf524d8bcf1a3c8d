"""Host logic of the replicas-only multi-GPU bench, run as two gloo ranks on
CPU: the barrier and the max-over-ranks timing reduction, that every replica
holds the same layer weights while drawing its own tokens, and the launch
path `bench.py --gpus N` takes when no launcher started it."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # each rank's "time" differs; the job time is the slowest rank's
        t = bench.max_over_ranks(10.0 + rank * 3.5, world, torch.device("cpu"))
        # replicas of one layer: identical weights, their own tokens
        from mixture_experts_layer_93_b300 import inputs as I
        cfg = I.MoEConfig("t", T=8, d=64, n=64, E=4, k=2)
        inp = I.make_replica_inputs(cfg, rank)
        out[rank] = (t, float(inp["x"].float().sum()), float(inp["W1"].float().sum()),
                     float(inp["Wr"].sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 13.5
    assert out[0][1] != out[1][1]                     # tokens differ
    assert out[0][2:] == out[1][2:]                   # weights and router agree


def test_bench_gpus_flag_launches_its_ranks():
    """`bench.py --gpus 2` (no WORLD_SIZE in the environment) starts two ranks
    itself; on the CPU they take gloo, and the dry run walks the replica
    set-up, the barrier and the max reduction the measured run uses."""
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--dry-run",
                          "--config", "tiny"], capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert res.returncode == 0, res.stderr[-3000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    j = json.loads(lines[0])
    assert j["n_gpus"] == 2 and j["max_rank_time"] == 2.0
    assert j["weights_identical"] is True and j["tokens_distinct"] is True
