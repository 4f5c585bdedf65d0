"""The multi-rank host logic of bench.py on CPU: two gloo ranks (one process
each), as torchrun would start them.  The whole-job time is the slowest
rank's, every rank sees the same value, the job's throughput counts every
rank's bytes (weak scaling), and the reference arm runs on rank 0 only."""
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) * 10 ms for the timed steps
        ms = bench.reduce_max(dist, 10.0 * (rank + 1))
        e2e = bench.reduce_max(dist, 3.0 - rank)
        args = type("A", (), {"steps": 2, "warmup": 3, "gpus": world})()
        buf = io.StringIO()
        if rank != 0:
            with redirect_stdout(buf):
                bench.run_reference(args, rank, world)
        out.put((rank, ms, e2e, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    assert [r[1] for r in res] == [20.0, 20.0]      # max over ranks
    assert [r[2] for r in res] == [3.0, 3.0]
    assert res[1][3] == ""                          # the reference arm prints nothing on rank 1




def test_job_throughput_counts_every_rank():
    one = bench.job_gbs(1, 821_133_332, 100, 17.77)
    assert abs(one - 821_133_332 * 100 / 17.77e-3 / 1e9) < 1e-9
    assert abs(bench.job_gbs(4, 821_133_332, 100, 17.77) - 4 * one) < 1e-6


def test_reduce_max_without_a_process_group_is_the_identity():
    assert bench.reduce_max(None, 12.5) == 12.5
