"""Host logic of the multi-GPU benchmark (replicas) on CPU gloo ranks."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    # rank r "took" 1 + r seconds for 10 * (r + 1) rows
    t, rows = bench.aggregate_ranks(1.0 + rank, 10 * (rank + 1), "cpu", dist)
    q.put((rank, t, rows))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_aggregate_is_max_time_and_summed_rows(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for _, t, rows in res:
        assert t == float(world)                      # slowest rank
        assert rows == float(sum(10 * (r + 1) for r in range(world)))


def test_single_rank_passthrough():
    import bench
    assert bench.aggregate_ranks(2.5, 7, "cpu", None) == (2.5, 7.0)
