"""The multi-rank path of bench.py on CPU (gloo, world size 2): every rank runs an
independent replica, the step time is the maximum over ranks and the value counts the
tokens of all ranks.  No GPU and no data-path collective."""
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
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = 10.0 + 5.0 * rank            # rank 1 is the slow one
        ms = bench.max_over_ranks(ms_local, dist, torch.device("cpu"))
        dist.barrier()
        out[rank] = (ms, bench.whole_job_value(world, 1000, ms / 4))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    # 2 ranks x 1000 tokens per step, 15 ms / 4 steps per step
    assert res[0][1] == pytest.approx(2 * 1000 / (15.0 / 4 / 1000.0))


def test_single_rank_has_no_collective():
    assert bench.max_over_ranks(7.5, None, None) == 7.5
    assert bench.whole_job_value(1, 1000, 67.0) == pytest.approx(1000 / 0.067)
