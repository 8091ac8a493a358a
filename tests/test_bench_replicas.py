"""bench.py's multi-replica path on CPU (gloo, world size 2): the job time is
the max over ranks, the job rate counts every rank's units, and the reference
arm prints from rank 0 only (other ranks exit without work)."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r's per-stage times; the job sees the slowest rank per entry
        mine = [1.0 + rank, 5.0 - rank, 2.5]
        got = bench.max_over_ranks(mine, world)
        w, r, _ = bench._dist()

        class Args:
            steps, warmup = 1, 0

        buf = io.StringIO()
        with redirect_stdout(buf):
            if r != 0:
                bench.run_reference(Args, w, r)  # returns at once on ranks > 0
        q.put((rank, got, w, r, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_max_and_only_rank0_prints():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, w, r, out in res:
        assert got == [2.0, 5.0, 2.5]
        assert (w, r) == (world, rank)
        assert out == ""
    assert bench.job_throughput(world, 3.0, 2.0) == 3.0
    assert bench.max_over_ranks([1.0, 2.0], 1) == [1.0, 2.0]

