"""What bench.py does at N > 1, on CPU (gloo, world size 2).

The path shards as independent replicas: every rank runs the whole workload
on its own GPU, with no data-path collective. The only cross-rank steps are
the timing reduction (the slowest rank's time, max over ranks) and the
whole-job throughput (world x one rank's bytes over that time). The reference
arm runs on rank 0 alone, which prints the one JSON line; the other ranks exit
0 without work."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank 1 is the slow one for the decode phase, rank 0 for the prefill
    local = {"dec_s": 0.010 + 0.005 * rank, "pre_ms": 3.0 - rank, "step_ms": 13.0 + 4.0 * rank, "wall": 1.0}
    timing = bench.reduce_max_over_ranks(local, world)
    value = bench.replica_throughput(1.0e9, timing["dec_s"], world)
    dist.destroy_process_group()
    q.put((rank, timing, value))


def test_two_replicas_max_timing_and_whole_job_throughput():
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
    (_, t0, v0), (_, t1, v1) = res
    want = {"dec_s": 0.015, "pre_ms": 3.0, "step_ms": 17.0, "wall": 1.0}
    for k, v in want.items():
        assert abs(t0[k] - v) < 1e-12 and abs(t1[k] - v) < 1e-12
    # 2 replicas x 1 GB each in the slowest rank's 15 ms
    assert abs(v0 - 2.0e9 / 0.015 / 1e9) < 1e-9 and v0 == v1


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    local = {"dec_s": 0.25, "wall": 2.0}
    assert bench.reduce_max_over_ranks(local, 1) == local
    assert abs(bench.replica_throughput(5.0e9, 0.25, 1) - 20.0) < 1e-12


def test_reference_arm_under_torchrun_prints_one_line():
    """bench.py --impl reference launched as the N = 2 runs are (torchrun, one
    process per rank): rank 0 prints one JSON line, rank 1 prints nothing, both
    exit 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1", "--config", "tiny_fp32"]
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 2
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
