"""Multi-rank path of bench.py on CPU: two gloo ranks, replica timing aggregation.

The decode path shards by (request, kv head) with no exchange, so N GPUs run N independent
replicas; the only cross-rank steps are the barrier and the max of the per-step time over ranks,
from which the whole-job throughput is formed.  These run here with the gloo backend.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [2.0, 3.5][rank]
        got = bench.rank_max(ms, torch.device("cpu"))
        dist.barrier()
        q.put((rank, got, bench.replica_throughput(world, 1e9, got)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [3.5, 3.5]
    # 2 replicas x 1 GB per step in 3.5 ms (the slowest rank)
    assert res[0][2] == pytest.approx(2 * 1e9 / 3.5e-3 / 1e9)


def test_single_process_is_identity():
    import torch
    import bench
    assert bench.rank_max(1.25, torch.device("cpu")) == 1.25
    assert bench.replica_throughput(1, 5e8, 0.5) == pytest.approx(1000.0)
