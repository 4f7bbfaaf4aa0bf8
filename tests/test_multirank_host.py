"""The multi-rank path of bench.py on the CPU: replicas over a gloo process
group of world size 2.  Each rank times its own copy of the work; the job's
time is the slowest rank's, and the job's rate counts every rank's units.
No GPU is involved (the GPU arm runs the same helpers over NCCL)."""
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank, world, port, queue):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    # Rank r's timings differ, as they would on two GPUs.
    times = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 3.0], world)
    rate = bench.job_throughput(100.0, world, times[0])
    dist.barrier()
    queue.put((rank, times, rate))
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_count_every_rank():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_replica, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, times, rate in results:
        assert times == [2.0, 10.0, 3.0], (rank, times)      # max over both ranks
        assert rate == 2 * 100.0 / 2.0                          # units of both ranks


def test_single_rank_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2], 1) == [1.5, 2.0]
    assert bench.job_throughput(10.0, 1, 4.0) == 2.5


def test_reference_arm_runs_on_rank_zero_only():
    # Under torchrun the reference arm's other ranks exit 0 without work.
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                         text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == ""
