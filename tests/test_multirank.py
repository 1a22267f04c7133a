"""The N>1 host path of bench.py with two gloo ranks on the CPU: every rank gets
the slowest rank's time and the job value sums the replicas; only rank 0 of the
reference arm does work."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.reduce_max_time(10.0 + 5.0 * rank, world, torch.device("cpu"))
    dist.barrier()
    w, r, _ = bench.dist_env()
    q.put((rank, ms, bench.job_value(world, 1e12, ms, 10), w, r))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value, w, r in out:
        assert ms == 15.0                       # the slower rank's time, on both ranks
        assert value == pytest.approx(2 * 1e12 / 1.5 / 1e9)  # two replicas of 1 TFLOP per 1.5 ms step
        assert (w, r) == (2, rank)


def test_reference_arm_nonzero_rank_does_nothing(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    from precision_grouped_gemm_gb300 import workloads as wl
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup, gpus = 1, 0, 2
    bench.run_reference(A, wl.DSV4_BF16)
    assert capsys.readouterr().out == ""
