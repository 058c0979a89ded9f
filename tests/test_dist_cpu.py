"""The multi-GPU path is replicas only: the bench's host-side helpers (barrier,
max over ranks, whole-job throughput) checked with two gloo ranks on CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        ms = [2.0, 3.5][rank]                       # rank 1 is the slow one
        mx = bench.reduce_max(ms, world, device="cpu")
        out[rank] = (mx, bench.job_throughput(1e9, mx, world))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == res[1][0] == 3.5
    # 2 ranks x 1 GB per step in 3.5 ms
    assert res[0][1] == pytest.approx(2e9 / 3.5e-3 / 1e9)


def test_single_rank_helpers():
    assert bench.reduce_max(1.25, 1) == 1.25
    assert bench.job_throughput(3.9e9, 0.6, 1) == pytest.approx(6500.0)
