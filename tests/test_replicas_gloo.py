"""The N > 1 path of bench.py without a GPU: two gloo ranks on the CPU.

Each rank runs an independent replica (the GEMM does not shard across
GPUs), so the only cross-rank steps are the barrier and the max over ranks
of the time per step; the whole-job value sums the ranks' work over the
slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, ms_by_rank, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, rank, world)
        bench.barrier(world)
        value, ms = bench.replica_throughput(2e12, ms_by_rank[rank], world)
        q.put((rank, value, ms))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    ms_by_rank = [1.0, 4.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, ms_by_rank, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = sorted(q.get(timeout=10) for _ in range(world))
    for rank, value, ms in results:
        assert ms == 4.0                       # max over ranks
        assert value == pytest.approx(world * 2e12 / 4e-3 / 1e12)  # both ranks' work / slowest time


def test_single_rank_needs_no_process_group():
    import bench
    value, ms = bench.replica_throughput(1e12, 2.0, 1)
    assert ms == 2.0 and value == pytest.approx(0.5e3)
