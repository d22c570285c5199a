"""The N > 1 path of bench.py on CPU: world-size-2 gloo ranks (replicas).

The library runs one GPU per process and its ranks never exchange data; what
spans ranks is the harness: process-group start-up, the barrier around the
timed region, the maximum of the per-rank step times, the whole-job rate, and
the reference arm, which only rank 0 runs."""
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), Q8_BENCH_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import io
    import contextlib
    import types

    import torch.distributed as dist

    import bench
    try:
        w, r, _ = bench.dist_init()
        # per-rank step times differ; every rank must see the slowest
        ms = bench.max_over_ranks(w, 1.0 + 0.5 * r)
        bench.barrier(w)
        rate = bench.aggregate_gbps(w, 1e9, ms)
        # the reference arm: rank 0 alone does work and prints
        args = types.SimpleNamespace(warmup=0, steps=0, gpus=w)
        out = io.StringIO()
        printed = None
        if r != 0:
            with contextlib.redirect_stdout(out):
                bench.run_reference(args, w, r)
            printed = out.getvalue()
        bench.barrier(w)
        q.put((r, w, ms, rate, printed))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, "error", repr(e), None, None))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_two_rank_replicas_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    world, port = 2, _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    try:
        for _ in range(world):
            r, w, ms, rate, printed = q.get(timeout=120)
            assert w != "error", ms
            res[r] = (w, ms, rate, printed)
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    assert sorted(res) == [0, 1]
    for r, (w, ms, rate, _) in res.items():
        assert w == 2
        assert ms == pytest.approx(1.5)                 # max over ranks
        assert rate == pytest.approx(2 * 1e9 / 1.5e-3 / 1e9)
    assert res[1][3] == ""                              # rank 1: reference arm silent
    assert all(p.exitcode == 0 for p in procs)


def test_single_process_defaults(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.max_over_ranks(1, 3.25) == 3.25
    assert bench.aggregate_gbps(1, 2e9, 2.0) == pytest.approx(1000.0)
    bench.barrier(1)   # no process group: a no-op
