"""Host logic of bench.py's N > 1 launch, on CPU: two ranks over gloo agree on the slowest
rank's step time, the whole-job value counts every replica's bytes, and the reference arm's
non-zero ranks exit without work.  (The path shards by replica: no collective on the data
path, only this timing reduction.)"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(dist, 1.0 + 0.5 * rank, "cpu")  # rank r took 1 + r/2 ms
        dist.barrier()
        q.put((rank, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_ranks_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=5) for _ in range(world))
    assert got == {0: 1.5, 1: 1.5}


def test_job_value_counts_every_replica():
    import bench
    one = bench.job_value(1, 71.3e6, 0.02)
    assert one == pytest.approx(71.3e6 / 20e-6 / 1e9)
    assert bench.job_value(4, 71.3e6, 0.02) == pytest.approx(4 * one)


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
