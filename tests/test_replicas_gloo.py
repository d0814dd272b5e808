"""The multi-GPU layout is replicas only: every rank decodes its own sequences on its own
model copy and the process group carries nothing but the start/stop barriers and the
timing reduction.  These run that host logic as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    r, w, local = bench.dist_setup(world, backend="gloo")
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    # rank r processed 10 * (r + 1) units in (r + 1) seconds
    value, dt = bench.aggregate(10.0 * (rank + 1), float(rank + 1), w)
    out.put((rank, value, dt, bench.max_over_ranks(float(rank), w), bench.sum_over_ranks(1.0, w)))
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replica_timing_is_total_units_over_slowest_rank(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    total = sum(10.0 * (r + 1) for r in range(world))
    slowest = float(world)
    for rank, value, dt, mx, n in res:
        assert dt == slowest
        assert value == pytest.approx(total / slowest)
        assert mx == world - 1
        assert n == world


def test_single_process_needs_no_group():
    assert bench.aggregate(64.0, 2.0, 1) == (32.0, 2.0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
