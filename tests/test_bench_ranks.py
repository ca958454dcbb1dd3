"""Host logic of bench.py's multi-GPU mode on CPU: two gloo ranks, each with its own timing, must
agree on the slowest rank's time and report whole-job (weak-scaling) throughput from it."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [120.0, 150.0][rank]
    mx = bench.max_over_ranks(ms, torch.device("cpu"))
    out[rank] = (mx, bench.whole_job_tflops(3.0e14, world, mx))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == res[1][0] == 150.0
    assert res[0][1] == pytest.approx(2 * 3.0e14 / 0.150 / 1e12)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(42.0, torch.device("cpu")) == 42.0
    assert bench.whole_job_tflops(1e12, 1, 1000.0) == pytest.approx(1.0)

