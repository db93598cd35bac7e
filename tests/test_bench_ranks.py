"""The benchmark's multi-rank plumbing (one process per GPU under torchrun) on CPU: two gloo
ranks take the max of their timings, pass the barriers and shut down; only rank 0 prints the
reference line.  The attention path shards by sequence with no collective (replicas), so this is
the only cross-rank logic."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    bench.ranks_init(world, backend="gloo")
    bench.ranks_barrier(world)
    mine = [1.0 + rank, 10.0 - rank, 5.0]
    got = bench.ranks_max(mine, world)
    bench.ranks_barrier(world)
    bench.ranks_done(world)
    queue.put((rank, got))


def test_two_gloo_ranks_take_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[0] == out[1] == [2.0, 10.0, 5.0]


def test_single_rank_is_the_identity():
    import bench
    assert bench.ranks_max([3.0, 4.0], 1) == [3.0, 4.0]
    bench.ranks_barrier(1)
    bench.ranks_done(1)


def test_reference_arm_prints_on_rank_0_only(capsys):
    import argparse

    import bench
    args = argparse.Namespace(workload="tiny", steps=1, warmup=0)
    bench.run_reference(args, rank=1, world=2)
    assert capsys.readouterr().out == ""
