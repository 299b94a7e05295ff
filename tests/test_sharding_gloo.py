"""Host logic of runs on several GPUs, exercised with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from latent_kv_cache_decode_b300.sharding import batch_shard, max_over_ranks


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        idx = batch_shard(8, world, rank)
        got = [None] * world
        dist.all_gather_object(got, idx)
        # rank r reports step time 1 + r: every rank must see the slowest one
        slowest = max_over_ranks(1.0 + rank, dist)
        q.put((rank, got, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_partition_batch_and_take_max_time():
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
    for rank, got, slowest in res:
        flat = sorted(i for shard in got for i in shard)
        assert flat == list(range(16))             # every global element exactly once
        assert slowest == 2.0


def test_shard_bounds():
    assert batch_shard(8, 1, 0) == list(range(8))
    assert batch_shard(8, 4, 3) == list(range(24, 32))
    with pytest.raises(ValueError):
        batch_shard(8, 2, 2)
    assert max_over_ranks(3.5) == 3.5
