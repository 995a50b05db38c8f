"""The benchmark's multi-GPU path is replicas only: each rank decodes its own
sequences (decode shards by sequence with no exchange step), the job's time
is the slowest rank's, and the job's throughput is every rank's bytes over
that time.  This checks that host logic with two gloo ranks on the CPU."""
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
    import bench
    mine = [1.0 + rank, 10.0 - rank, 0.5 * (rank + 1)]        # per-rank times
    got = bench.max_over_ranks(mine)
    value = bench.whole_job_gbs(world, 4_000_000_000, got[0])
    q.put((rank, got, value))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in res:
        assert got == [2.0, 10.0, 1.0]                    # max over both ranks, element-wise
        assert value == pytest.approx(2 * 4.0 / 2.0e-3)    # 2 ranks x 4 GB over 2 ms, in GB/s


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
    assert bench.whole_job_gbs(1, 1_000_000_000, 1.0) == pytest.approx(1000.0)
