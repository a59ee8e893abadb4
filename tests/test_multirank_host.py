"""The N>1 bench path on the host: two gloo ranks (CPU), each timing its own
replica; rank 0 must see the slowest rank's time and the job-wide value."""
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
    ws, r, _ = bench.dist_env()
    assert (ws, r) == (world, rank)
    my_ms = 100.0 + 50.0 * rank          # rank 1 is the slow one
    worst = bench.max_over_ranks(my_ms, ws, device="cpu")
    bench.barrier(ws)
    q.put((rank, worst))
    dist.destroy_process_group()


def test_two_rank_max_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(world))
    assert got == {0: 150.0, 1: 150.0}


def test_flop_convention():
    import bench
    from seeded_inputs import WORKLOADS
    w = WORKLOADS["train_s32k"]
    assert bench.flops(w, bwd=False) == pytest.approx(4.398e12, rel=1e-3)     # 2 B H S^2 D
    assert bench.flops(w, fwd=False) == pytest.approx(10.995e12, rel=1e-3)    # 5 B H S^2 D
    assert bench.flops(WORKLOADS["fwd_s8k"]) == pytest.approx(274.9e9, rel=1e-3)
