"""Request sharding and the cross-rank timing reduction, on CPU with two gloo ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from semi_ar_draft_gb300 import shard


def test_shards_cover_the_batch_once():
    for B in (0, 1, 7, 32, 33, 512):
        for world in (1, 2, 3, 8):
            seen = []
            sizes = []
            for rank in range(world):
                s, n = shard.shard_requests(B, world, rank)
                seen.extend(range(s, s + n))
                sizes.append(n)
            assert seen == list(range(B))
            assert max(sizes) - min(sizes) <= 1


def test_bad_rank_is_rejected():
    with pytest.raises(ValueError):
        shard.shard_requests(8, 2, 2)
    with pytest.raises(ValueError):
        shard.shard_requests(8, 0, 0)


def test_rank_seeds_differ_and_keep_low_word():
    seeds = {shard.rank_seed(12345, r) for r in range(8)}
    assert len(seeds) == 8
    assert all((s & 0xFFFFFFFF) == 12345 for s in seeds)
    assert shard.rank_seed(2 ** 64 - 1, 1) == (2 ** 64 - 1 + 2 ** 32) % 2 ** 64


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        start, n = shard.shard_requests(33, world, rank)
        # a rank's "step time" grows with its shard; the job time is the slowest rank's
        t_local = 0.001 * (n + rank)
        t = shard.max_over_ranks(t_local, dist)
        counts = torch.tensor([n], dtype=torch.int64)
        dist.all_reduce(counts)
        out[rank] = (start, n, t, int(counts.item()), shard.job_throughput(n, world, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs)
        res = dict(out)
    (s0, n0, t0, c0, _), (s1, n1, t1, c1, _) = res[0], res[1]
    assert (s0, n0, s1, n1) == (0, 17, 17, 16)
    assert c0 == c1 == 33
    slowest = max(0.001 * (17 + 0), 0.001 * (16 + 1))
    assert t0 == t1 == pytest.approx(slowest)
    # whole-job throughput: each rank's units over the slowest time
    assert shard.job_throughput([n0, n1], world, t0) == pytest.approx(33 / slowest)
