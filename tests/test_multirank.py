"""Multi-rank host logic of bench.py on CPU: two gloo ranks.

The draft path is data-parallel over independent sequences (replicas, no
collective on the data path); what spans ranks is the timing protocol: every
rank times its own replica, the slowest rank's time is taken with a MAX
all-reduce, and the whole-job rate counts the units of all ranks over that
time.  Rank 0 alone prints; the reference arm runs on rank 0 only.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 5.0 * rank  # rank 1 is the slower replica
    slowest = bench.max_over_ranks(local_ms, world)
    rate = bench.whole_job_rate(world, 3, 100, slowest)
    dist.barrier()
    out.put((rank, slowest, rate))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_all_units():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    for _, slowest, rate in res:
        assert slowest == 15.0
        # 2 ranks x 3 sequences x 100 steps in 15 ms
        assert rate == pytest.approx(2 * 3 * 100 / 0.015)


def test_single_rank_is_a_no_op():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.25, 1) == 7.25
    assert bench.whole_job_rate(1, 1, 1000, 500.0) == pytest.approx(2000.0)


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup = 1, 0

    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(Args, rank=1, world=2)
    assert buf.getvalue() == ""
