"""The benchmark's multi-rank logic on CPU: two gloo ranks, each a replica with its own
step time; the job's time is the slowest rank's and the throughput counts every rank's
work (weak scaling, no collective on the data path)."""
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
    import bench
    my_ms = [10.0, 25.0][rank]                      # rank 1 is the slow one
    total = bench.reduce_max(my_ms, world)
    agg = bench.aggregate(per_rank_bytes=1e9, per_rank_seqs=64, max_ms_total=total, world=world, steps=5)
    q.put((rank, total, agg))
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_aggregate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, agg in res:
        assert total == 25.0                          # the slowest rank sets the time
        assert agg["ms_per_step"] == pytest.approx(5.0)
        # 2 ranks x 5 steps x 1 GB in 25 ms = 400 GB/s; 2 x 5 x 64 sequences
        assert agg["gbs"] == pytest.approx(400.0)
        assert agg["seqs_per_s"] == pytest.approx(2 * 5 * 64 / 0.025)
