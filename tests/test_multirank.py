"""bench.py's multi-GPU path is one independent replica per rank (the hot path
has no exchange step): the job's step time is the slowest rank's, and its
throughput is the units of all ranks over that time.  Checked here with two
gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    step = [0.010, 0.013][rank]
    slowest = bench.slowest_rank_seconds(step, dist, torch.device("cpu"))
    value = bench.replica_throughput(5.0e8, world, slowest)
    q.put((rank, slowest, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for _, slowest, value in res:
        assert slowest == pytest.approx(0.013)
        assert value == pytest.approx(2 * 5.0e8 / 0.013)


def test_single_process_is_unchanged():
    import bench
    assert bench.slowest_rank_seconds(0.02, None) == 0.02
    assert bench.replica_throughput(10.0, 1, 2.0) == 5.0
