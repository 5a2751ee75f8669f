"""The bench's multi-GPU host logic (independent replicas, one process per GPU) on CPU.

Two gloo ranks stand in for two GPUs: the barrier, the max over ranks of the timed
seconds and the whole-job throughput (every rank's tokens over the slowest rank's time)
are the same code the NCCL run uses.
"""
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
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    d = bench.Dist(world, backend="gloo")
    d.barrier()
    seconds = 0.5 + rank          # rank 1 is the slower replica
    slowest = d.max(seconds)
    out[rank] = (d.world, slowest, bench.aggregate_throughput(4, 10, d.world, slowest))
    d.barrier()
    d.pg.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(2):
        world, slowest, value = res[r]
        assert world == 2 and slowest == pytest.approx(1.5)
        assert value == pytest.approx(4 * 10 * 2 / 1.5)


def _graph_rank(rank, world, port, fail_rank, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    d = bench.Dist(world, backend="gloo")
    failed = rank == fail_rank
    res = bench.graph_result(d, float("inf") if failed else 0.002 * (rank + 1), "capture refused" if failed else None,
                             8, 100)
    out[rank] = res
    d.barrier()
    d.pg.destroy_process_group()


@pytest.mark.parametrize("fail_rank", [-1, 1])
def test_graph_figure_needs_every_rank(fail_rank):
    """Every rank joins the max over ranks, also one whose graph capture failed, so no rank waits
    for a collective that another rank skipped; the figure stands only if all captures worked."""
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_graph_rank, args=(r, 2, port, fail_rank, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    if fail_rank < 0:
        for r in range(2):
            assert res[r]["us_per_layer"] == pytest.approx(0.004 / 100 * 1e6)
            assert res[r]["value"] == pytest.approx(8 * 100 * 2 / 0.004)
    else:
        assert res[1] == {"error": "capture refused"}
        assert res[0] == {"error": "graph capture failed on another rank"}


def test_single_process_needs_no_group():
    d = bench.Dist(1, backend="gloo")
    assert d.world == 1 and d.max(3.0) == 3.0
    assert bench.aggregate_throughput(1, 200, 1, 0.004) == pytest.approx(50000.0)
