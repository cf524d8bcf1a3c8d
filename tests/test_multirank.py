"""Host logic of the replicas-only multi-GPU bench, run as two gloo ranks on
CPU: the barrier and the max-over-ranks timing reduction, and that each
rank's replica is independent (no data-path collective)."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # each rank's "time" differs; the job time is the slowest rank's
        t = bench.max_over_ranks(10.0 + rank * 3.5, world, torch.device("cpu"))
        # replicas draw their own inputs (seed = rank): no exchange needed
        from mixture_experts_layer_93_b300 import inputs as I
        cfg = I.MoEConfig("t", T=8, d=64, n=64, E=4, k=2)
        x = I.make_inputs(cfg, seed=rank, weights=False)["x"]
        out[rank] = (t, float(x.float().sum()))
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
    assert out[0][1] != out[1][1]
