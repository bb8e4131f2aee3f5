"""bench.py's multi-rank host logic with two gloo ranks on the CPU: rank discovery from the
environment, the barrier, max-over-ranks timing, and the whole-job value of weak scaling."""

from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    r, w, local = bench.dist_init("gloo")
    try:
        bench.barrier(w)
        # each rank "measured" a different step time; the slowest one counts
        mine = 1.0 + rank
        worst = bench.max_over_ranks(mine, w)
        value = bench.job_value(units_per_rank=262144, world=w, seconds_max=worst * 1e-3)
        q.put((r, w, local, worst, value))
    finally:
        import torch.distributed as dist
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 for r in res)
    assert all(r[3] == 2.0 for r in res)  # max over ranks seen by both
    # whole job: 2 ranks x 262144 query-heads in 2 ms
    assert all(abs(r[4] - 2 * 262144 / 2e-3) < 1e-6 for r in res)


def test_single_rank_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_value(10, 1, 2.0) == 5.0
