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



def _owned_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import workloads
    shapes = workloads.llama3_8b_shapes(32)
    mine = bench.owned_shapes(shapes, world, rank)
    names = [None] * world
    dist.all_gather_object(names, [n for n, _, _ in mine])
    flops = bench.total_flops(mine, "gram")
    ms = flops / 1.5e12  # this rank's step time at 1.5 PFLOP/s (ms)
    mx = bench.max_over_ranks(ms, torch.device("cpu"))
    out[rank] = (names, flops, mx)
    dist.barrier()
    dist.destroy_process_group()


def test_owned_mode_splits_the_set_across_ranks():
    """bench.py --owned: each rank computes its share on its own (dmuon_assign_owners, no communication);
    the shares cover every matrix of the 224-matrix set exactly once, and the job's time is the slowest
    rank's, so the whole-job rate is the set's flops over that time (strong scaling)."""
    import bench
    import workloads
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_owned_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=300)
            assert p.exitcode == 0
        res = dict(out)
    shapes = workloads.llama3_8b_shapes(32)
    names = res[0][0]
    assert names == res[1][0]
    flat = [n for share in names for n in share]
    assert sorted(flat) == sorted(n for n, _, _ in shapes) and len(flat) == len(set(flat))
    total = bench.total_flops(shapes, "gram")
    assert res[0][1] + res[1][1] == total
    slowest = max(res[0][1], res[1][1]) / 1.5e12
    assert res[0][2] == res[1][2] == pytest.approx(slowest)
    assert max(res[0][1], res[1][1]) / (total / world) < 1.05  # LPT balance
