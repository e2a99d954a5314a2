"""The multi-rank logic of bench.py on the CPU: two gloo ranks.

With N GPUs every rank runs its own replica of the scan (rows are independent,
so there is no exchange step); the job's time is the slowest rank's timed
region and its throughput counts the units of all ranks. These tests run that
host-side aggregation with the gloo backend, no GPU involved."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, timed_ms, queue):
    import torch
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.max_over_ranks(dist, timed_ms[rank], torch.device("cpu"))
        v = bench.replica_throughput(world, 1000, 4, m)
        queue.put((rank, m, v))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_sum_the_work():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    timed_ms = [10.0, 15.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, timed_ms, queue)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = sorted(queue.get(timeout=120) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, m, v in results:
        assert m == 15.0, (rank, m)
        assert v == pytest.approx(2 * 1000 * 4 / 15e-3, rel=1e-12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(None, 12.5, None) == 12.5
    assert bench.replica_throughput(1, 1000, 4, 12.5) == pytest.approx(1000 * 4 / 12.5e-3)


def test_reference_arm_other_ranks_exit_without_work():
    """Under torchrun only rank 0 times the oracle and prints; the others return."""
    import bench
    out = io.StringIO()
    with redirect_stdout(out):
        assert bench.run_reference(None, 1, 2) is None
    assert out.getvalue() == ""
