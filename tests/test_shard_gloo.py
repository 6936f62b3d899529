"""Multi-rank host logic on CPU: two gloo ranks shard sequences and agree on the job time."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from looped_normalized_gpt_gb300.shard import job_throughput, shard


def test_shards_cover_every_sequence_once():
    for n in (1, 7, 16, 64, 65):
        for world in (1, 2, 3, 8):
            seen = [i for r in range(world) for i in shard(n, r, world)]
            assert seen == list(range(n))
            sizes = [len(shard(n, r, world)) for r in range(world)]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard(4, 2, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    import torch.distributed as dist

    from looped_normalized_gpt_gb300.shard import shard as sh, slowest

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = list(sh(64, rank, world))
        dist.barrier()
        ms = slowest(10.0 + 5.0 * rank)  # rank 1 is the slow one
        q.put((rank, mine, ms))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, t0), (r1, s1, t1) = out
    assert t0 == t1 == 15.0
    assert set(s0).isdisjoint(s1) and sorted(s0 + s1) == list(range(64))
    assert job_throughput([len(s0), len(s1)], t0, 2) == pytest.approx(64 / 0.015)
