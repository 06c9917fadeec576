"""Host logic of multi-rank runs on CPU (gloo, world size 2): requests are
sharded as independent replicas with no data-path collective, and a run's
timing is the max over ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import bench
    import workload
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    shard = workload.shard_requests(130, rank, world)
    timing = bench.reduce_max_over_ranks({"step_ms": 10.0 + rank, "wall": 1.0 * (2 - rank)}, world)
    dist.destroy_process_group()
    q.put((rank, shard, timing))


def test_two_rank_sharding_and_max_timing():
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
    (_, s0, t0), (_, s1, t1) = res
    assert s0 + s1 == list(range(130)) and abs(len(s0) - len(s1)) <= 1
    assert t0 == t1 == {"step_ms": 11.0, "wall": 2.0}


@pytest.mark.parametrize("n,world", [(16, 1), (16, 3), (5, 8), (0, 2)])
def test_shard_requests_partition(n, world):
    import workload
    got = [workload.shard_requests(n, r, world) for r in range(world)]
    assert sum(got, []) == list(range(n))
