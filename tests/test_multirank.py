"""The multi-process path of bench.py on CPU ranks (gloo, world size 2,
127.0.0.1): every rank receives the slowest rank's timings, the whole-job rate
counts the units of all ranks, and only rank 0 runs and prints the reference
arm.  One process per GPU is the deployment; the path has no data exchange
(independent replicas), so the timing reduction is the only collective."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r was slower on the first figure, faster on the second
        out = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 3.0], dist)
        q.put((rank, out))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_every_rank_gets_the_slowest_rank_timings():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert got == {0: [2.0, 10.0, 3.0], 1: [2.0, 10.0, 3.0]}


def test_alone_the_timings_pass_through():
    assert bench.max_over_ranks([0.5, 2]) == [0.5, 2.0]


def test_job_rate_counts_every_rank():
    assert bench.job_rate(1, 8192, 0.5) == pytest.approx(8192 / 0.5e-3)
    assert bench.job_rate(4, 8192, 0.5) == pytest.approx(4 * 8192 / 0.5e-3)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class Args:
        workload, steps, warmup = "tiny", 1, 0
    assert bench.run_reference(Args, rank=1, world=2) == 0
    assert capsys.readouterr().out == ""
