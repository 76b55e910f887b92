"""The multi-process (replica) path of bench.py on CPU: two gloo ranks.

With N GPUs every rank runs its own replica of the attention step (the path
has no exchange step); the job's time is the slowest rank's and its work is N
times one replica's.  These tests run that host logic with the gloo backend,
world size 2, and check the rank-0-only behaviour of the reference arm.
"""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_init()
        ms = [3.0, 5.0][r]  # rank 1 is the slower replica
        slow = bench.slowest_over_ranks(ms, w, "cpu")
        out.put((r, w, local, slow, bench.whole_job_tflops(w, 1e12, slow)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, world, local, slow, tflops) in enumerate(res):
        assert (rank, world, local) == (r, 2, r)
        assert slow == 5.0  # every rank sees the slowest rank's time
        # two replicas of 1e12 flops each in 5 ms: 400 TFLOP/s for the job
        assert tflops == pytest.approx(2 * 1e12 / 5e-3 / 1e12)


def test_single_process_needs_no_process_group():
    assert bench.slowest_over_ranks(7.5, 1, "cpu") == 7.5
    assert bench.whole_job_tflops(1, 2e12, 10.0) == pytest.approx(200.0)


def test_reference_arm_prints_only_on_rank_zero(capsys):
    class Args:
        steps, warmup, gpus = 1, 3, 2
    assert bench.run_reference(Args, world=2, rank=1) == 0
    assert capsys.readouterr().out == ""
