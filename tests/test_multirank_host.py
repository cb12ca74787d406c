"""Replica mode across ranks, on the CPU (gloo, world size 2).

The layer has no exchange step, so several GPUs run independent replicas: the
bench's step time is the slowest rank's (a max over the ranks), the job's rate
counts every replica's tokens, and the reference arm runs and prints on rank 0
only while the other ranks exit at once.
"""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _replica(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    ms = bench.max_over_ranks(1.0 + 0.5 * rank, world, torch.device("cpu"))
    rate = bench.job_rate(64, ms, world)
    torch.distributed.barrier()
    q.put((rank, ms, rate))
    torch.distributed.destroy_process_group()


def test_step_time_is_the_slowest_rank_and_rate_counts_every_replica():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_replica, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    assert [r[1] for r in res] == [1.5, 1.5]             # both ranks see the slower one
    for r in res:
        assert r[2] == pytest.approx(2 * 64 / 1.5e-3)    # two replicas' tokens over 1.5 ms


def test_one_rank_alone_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1, None) == 2.5
    assert bench.job_rate(64, 2.0, 1) == pytest.approx(32000.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""               # no result line from rank 1
