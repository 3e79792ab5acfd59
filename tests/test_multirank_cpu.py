"""World-size-2 gloo checks (CPU) of the bench's multi-rank host logic: the
units of a partitioned workload are split across ranks exactly once, and the
timed region is the maximum over ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        times = [10.0 + rank, 3.0 * (world - rank), 7.0]
        out[rank] = bench.reduce_max(times)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == [11.0, 6.0, 7.0]


def test_reduce_max_without_process_group_is_identity():
    assert bench.reduce_max([1.5, 2.5]) == [1.5, 2.5]


@pytest.mark.parametrize("total,world", [(0, 2), (1, 2), (7, 2), (1024, 2), (33, 4), (512, 8)])
def test_shard_units_partition(total, world):
    seen = []
    for r in range(world):
        part = bench.shard_units(total, r, world)
        assert len(part) in (total // world, total // world + 1)
        seen.extend(part)
    assert seen == list(range(total))
