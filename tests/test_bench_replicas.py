"""The N > 1 path of bench.py on CPU: two gloo ranks stand in for two GPUs.

Each rank is an independent replica (the step has no exchange), so the only
cross-rank work is the barrier, the maximum of the elapsed times and, for the
oracle arm, rank 0 alone doing the work.  These tests run that host logic in
two processes."""

import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        own_ms = [3.0, 5.0][rank]
        dist.barrier()
        ms = bench.max_over_ranks(own_ms, torch.device("cpu"))
        rate = bench.whole_job_rate(32 * 10, ms, world)

        class Args:
            steps, warmup = 1, 3

        ref_line = bench.reference_arm(Args, rank, world) if rank == 1 else "skipped"
        out.put((rank, ms, rate, ref_line))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = {}
    for _ in range(world):
        r, ms, rate, ref = q.get(timeout=120)
        results[r] = (ms, rate, ref)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank reports the slowest rank's time
    assert results[0][0] == results[1][0] == 5.0
    # whole-job rate: 2 ranks x 320 tokens in 5 ms
    assert results[0][1] == pytest.approx(2 * 320 / 5e-3)
    # the oracle arm runs on rank 0 only; other ranks return nothing
    assert results[1][2] is None
