"""bench.py's multi-rank bookkeeping with two gloo ranks on the CPU: the
barrier-bracketed maximum over ranks and the whole-job aggregate (replicas:
each rank quantizes its own batch, no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    mine = 10.0 + 5.0 * rank  # rank 1 is the slow one
    total = bench.max_over_ranks(mine, world, torch.device("cpu"))
    dist.barrier()
    out[rank] = total
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
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
        assert out[0] == out[1] == 15.0


def test_aggregate_counts_every_replica():
    b = bench.counted_bytes(bench.wl.WORKLOADS["act_rht_sr_8192x4096"])["total"]
    assert b == 153_092_104
    one = bench.aggregate_gbs(b, 0.05, 1)
    assert bench.aggregate_gbs(b, 0.05, 4) == pytest.approx(4 * one)
    assert bench.max_over_ranks(3.0, 1, torch.device("cpu")) == 3.0
