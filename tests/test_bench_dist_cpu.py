"""The multi-process (replicas) path of bench.py on the CPU: gloo, world size 2, rendezvous on 127.0.0.1."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r measured a step of 1 + r ms and an end-to-end step of 5 - r ms
    out = bench.max_over_ranks([1.0 + rank, 5.0 - rank], "cpu")
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, out))


def test_slowest_rank_sets_the_step_time_world2():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 5.0]


def test_job_throughput_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    flops = 2841.0e9  # one large-layer step
    one = bench.job_tflops(1, flops, 2.0)
    assert one == pytest.approx(1420.5)
    # two replicas, each with its own step of the same length: twice the work in the (max) time
    assert bench.job_tflops(2, flops, 2.0) == pytest.approx(2 * one)
    # a slower rank lowers the whole job's throughput
    assert bench.job_tflops(2, flops, 4.0) == pytest.approx(one)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"], env=env,
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
