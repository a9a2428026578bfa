"""The N > 1 path of bench.py on CPU: two gloo ranks on this host.

Under torchrun every rank runs an independent replica (the sequences are
independent: no data-path collective); the only cross-rank steps are the
barriers around the timed region and the max-over-ranks of the elapsed time.
These tests run those steps, and the reference arm's rank split, with
world_size 2 on the gloo backend.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    bench.init_dist(ws, "gloo")
    bench.barrier(ws)
    # each rank reports its own elapsed time; every rank must see the maximum
    got = bench.max_over_ranks(10.0 * (rank + 1), ws)
    bench.barrier(ws)
    out[rank] = got
    dist.destroy_process_group()


def _reference_rank(rank, world, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import io
    from contextlib import redirect_stdout

    import bench

    class Args:
        steps, warmup, gpus = 1, 3, world

    buf = io.StringIO()
    if rank == 0:
        out[rank] = "skipped"   # rank 0 would time the oracle (covered by the single-process tests)
        return
    with redirect_stdout(buf):
        bench.run_reference(Args())
    out[rank] = buf.getvalue()


def test_barrier_and_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == pytest.approx(20.0) and out[1] == pytest.approx(20.0)


def test_reference_arm_other_ranks_exit_without_work():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    p = ctx.Process(target=_reference_rank, args=(1, 2, out))
    p.start()
    p.join(timeout=120)
    assert p.exitcode == 0
    assert out[1] == ""   # only rank 0 prints the reference line
