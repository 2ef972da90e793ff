"""The N>1 path of bench.py on CPU: two gloo ranks, no GPU.

The op shards by sequence with no data-path exchange, so each rank draws its
own batch and the only cross-rank traffic is a barrier and the max / sum of
the per-rank timings and byte counts."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        cfg = bench.rank_config("batched_decode", rank)
        bench.barrier(world)
        t = bench.reduce_max(1.5 + rank, world)
        s = bench.reduce_sum(10.0 * (rank + 1), world)
        q.put((rank, cfg.seed, cfg.groups, t, s))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_by_seed_and_reduce_timings():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    (r0, seed0, g0, t0, s0), (r1, seed1, g1, t1, s1) = got
    assert seed0 != seed1 and g0 == g1 == 256          # same shape, independent batches
    assert t0 == t1 == 2.5                             # max over ranks
    assert s0 == s1 == 30.0                            # whole-job sum
