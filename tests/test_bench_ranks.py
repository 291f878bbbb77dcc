"""Multi-rank logic of bench.py on CPU (gloo, world size 2): the elapsed time
reported is the slowest rank's, the whole-job rate counts every rank's units,
and in the reference arm only rank 0 runs and prints."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.5, 4.0][rank]
        slowest = bench.max_over_ranks(mine, world, "cpu")
        rate = bench.job_throughput(world, 64, 10, slowest)
        buf = io.StringIO()

        class Args:  # the reference arm on a non-zero rank must do nothing
            steps, warmup = 3, 3
        if rank == 1:
            with redirect_stdout(buf):
                bench.run_reference(Args, rank, world)
        q.put((rank, slowest, rate, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_and_count_all_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, rate, printed in out:
        assert slowest == 4.0
        assert rate == pytest.approx(2 * 64 * 10 / 4.0)
        assert printed == ""


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1, "cpu") == 2.5
    assert bench.job_throughput(1, 64, 200, 0.5) == pytest.approx(25600.0)
