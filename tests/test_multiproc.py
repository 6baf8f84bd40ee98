"""Replica path of bench.py with world size 2 on the CPU (gloo), no GPU.

The hot path does not shard: each replica runs the whole cycle on its own
batch. What multi-process runs add is host logic: rank setup from the
launcher's environment, the barrier around the timed region, the max of the
per-rank times, and rank 0 alone printing (and alone running the reference
arm). These tests run that logic in two spawned processes.
"""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, ws, local = bench.dist_setup()
    assert dist.get_backend() == "gloo"
    bench.barrier(ws)
    t = bench.reduce_max(1.5 + r, ws)        # per-rank "times" 1.5 and 2.5
    # the reference arm runs on rank 0 only; other ranks return without work
    ran = None
    if r != 0:
        import io
        import contextlib
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            class A:
                workload, warmup, steps, gpus = "tiny_B4_K4_V1024", 0, 1, ws
            bench.run_reference(A, r, ws)
        ran = buf.getvalue()
    bench.barrier(ws)
    dist.destroy_process_group()
    q.put((r, ws, local, t, ran))


def test_two_rank_setup_barrier_and_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=240) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert [o[0] for o in out] == [0, 1]
    assert all(o[1] == 2 for o in out)
    assert all(o[3] == 2.5 for o in out)      # max over ranks, seen by every rank
    assert out[1][4] == ""                    # rank 1 printed nothing for the reference arm
