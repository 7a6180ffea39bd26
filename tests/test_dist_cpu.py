"""The benchmark's multi-rank plumbing on CPU: two gloo ranks (replicas only).

The path has no exchange step, so `bench.py --gpus N` runs N independent
replicas: a barrier on both sides of the timed region, the maximum of the
ranks' step times, and a whole-job value of N times one replica's bytes over
that maximum.  These tests run that host logic with world size 2 and no GPU.
"""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, step_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import bench
    r, w, local, dist = bench.dist_setup(world)
    try:
        bench.barrier(dist)
        ms = bench.max_over_ranks(dist, step_ms[rank])
        bench.barrier(dist)
        q.put((r, w, local, dist.get_backend(), ms, bench.job_value(w, 1.0e9, ms)))
    finally:
        dist.destroy_process_group()


def _run(world, step_ms):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, step_ms, q))
             for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out)


def test_two_replicas_take_the_slowest_rank():
    out = _run(2, [2.0, 5.0])
    assert [o[0] for o in out] == [0, 1]
    for r, w, local, backend, ms, value in out:
        assert w == 2 and local == r and backend == "gloo"
        assert ms == 5.0                               # max over ranks, on every rank
        assert value == pytest.approx(2 * 1.0e9 * 1e3 / 5.0 / 1e9)   # 400 GB/s


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    old = os.environ.pop("WORLD_SIZE", None)
    try:
        r, w, local, dist = bench.dist_setup(1)
    finally:
        if old is not None:
            os.environ["WORLD_SIZE"] = old
    assert (r, w, local, dist) == (0, 1, 0, None)
    bench.barrier(None)
    assert bench.max_over_ranks(None, 3.25) == 3.25
    assert bench.job_value(1, 122683392, 0.0344) == pytest.approx(3566.4, rel=1e-4)
