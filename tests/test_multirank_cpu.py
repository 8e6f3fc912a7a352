"""The benchmark's multi-process path on CPU (gloo, world size 2): the timed
region's slowest rank sets the job time, the whole-job rate counts every
rank's tokens, and the reference arm runs on rank 0 only.  Replicas only: the
hot path has no data exchange between ranks."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) * 10 ms: the job took the slowest rank's 20 ms
        t = bench.max_over_ranks(dist, (rank + 1) * 10.0, torch.device("cpu"))
        rate = bench.job_rate(world, 16384, 4, t)
        # the reference arm: rank 0 alone runs and prints, the others return
        buf = io.StringIO()

        class A:
            steps, warmup, gpus = 1, 0, world
        if rank != 0:
            with redirect_stdout(buf):
                bench.run_reference(A, None)
        out.put((rank, t, rate, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_time_and_whole_job_rate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(world))
    for rank, t, rate, printed in res:
        assert t == 20.0
        assert rate == pytest.approx(world * 16384 * 4 / 0.020)
        if rank != 0:
            assert printed == ""


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 12.5, None) == 12.5
    assert bench.job_rate(1, 1000, 10, 1000.0) == pytest.approx(10000.0)
