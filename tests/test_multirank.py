"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): the slowest
rank's time is what every rank reports, and sharding a batch of independent
sequences over ranks covers every sequence exactly once, with no data-path
collective."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        t = bench._max_over_ranks(1.0 + rank * 0.5, True)
        q.put((rank, t, list(bench.shard_of(37, rank, world))))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_shard_disjointly():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(t == 1.5 for _, t, _ in res)
    units = sorted(u for _, _, shard in res for u in shard)
    assert units == list(range(37))


def test_shard_of_single_rank_is_everything():
    import bench
    assert list(bench.shard_of(5, 0, 1)) == list(range(5))
    assert [len(bench.shard_of(10, r, 3)) for r in range(3)] == [3, 3, 4]
