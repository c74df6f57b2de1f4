"""The multi-GPU path of the benchmark is replicas only (batch-1 decode has
no units to shard without a per-layer all-reduce): each rank decodes its own
copy and the job's time is the slowest rank's.  These tests run that
aggregation with two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(times[rank], dist, "cpu")
        out.put((rank, ms, bench.replica_throughput(world, 10, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [12.5, 20.0]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tps in res:
        assert ms == 20.0                       # every rank sees the slowest rank's time
        assert tps == pytest.approx(2 * 10 / 0.020)   # whole-job tokens/s over both replicas


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.0, None, "cpu") == 7.0
    assert bench.replica_throughput(1, 256, 500.0) == pytest.approx(512.0)
