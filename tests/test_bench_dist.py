"""The benchmark's multi-rank timing logic on CPU: two gloo ranks.

Each rank measures its own time; the job's time is the slowest rank's and
the throughput counts the bytes of every rank (weak scaling, no data-path
collective)."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    local_ms = 10.0 + 5.0 * rank                      # rank 1 is the slower one
    mx = bench.reduce_max_over_ranks(local_ms)
    out[rank] = (r, w, lr, mx, bench.job_throughput(1e9, w, 100, mx))
    dist.destroy_process_group()


def test_two_rank_timing_aggregation():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        rr, w, lr, mx, gbs = out[r]
        assert (rr, w, lr) == (r, 2, r)
        assert mx == pytest.approx(15.0)                  # the slowest rank
        assert gbs == pytest.approx(1e9 * 2 * 100 / 15e-3 / 1e9)


def test_single_process_is_identity():
    assert bench.reduce_max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(2e9, 1, 10, 1000.0) == pytest.approx(20.0)
