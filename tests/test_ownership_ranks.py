"""Dedicated ownership across ranks, on CPU with two gloo ranks (DMuon "Core Concepts", section "1.
Dedicated Ownership"; section "均衡划分" for the LPT rule). Every rank computes the owner map on its own
with dmuon_assign_owners and no communication; the maps must agree, give each matrix exactly one owner,
and report per-rank loads equal to the summed cost of the matrices each rank owns. Each rank then
updates only the matrices it owns (float64 oracle) and the updates are exchanged: the assembled result
must equal a single process updating every matrix, bit for bit."""

import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

import newton_schulz_momentum_gb300 as dm
import workloads
from newton_schulz_momentum_gb300 import build as dmbuild

WORLD = 2
TINY = [(8, 16), (16, 8), (12, 12), (4, 20), (20, 4), (10, 30), (6, 6), (24, 8)]
TINY_LAYERS = [0, 0, 0, 1, 1, 1, 2, 2]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _tiny_inputs(i, shape):
    w0 = workloads.gaussian(shape, 0.02, 300 + i).astype(np.float64)
    g = workloads.gaussian(shape, 1.0, 400 + i).astype(np.float64)
    return w0, g, np.zeros(shape)


def _worker(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(WORLD))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    from oracle import ns64

    shapes = [(r, c) for _, r, c in workloads.llama3_8b_shapes(32)]
    layers = [i // 7 for i in range(len(shapes))]
    owners, loads = dm.assign_owners(shapes, WORLD, layers, "gram_flops")
    maps = [None] * WORLD
    dist.all_gather_object(maps, (owners, loads))

    tiny_owners, _ = dm.assign_owners(TINY, WORLD, TINY_LAYERS, "gram_flops")
    mine = {}
    for i, s in enumerate(TINY):
        if tiny_owners[i] == rank:
            w0, g, m0 = _tiny_inputs(i, s)
            r = ns64.muon_step(w0, g, m0, 0.02, 0.95, ns64.YOU, (2,), "gram")
            mine[i] = (r["W"], r["M"])
    gathered = [None] * WORLD
    dist.all_gather_object(gathered, mine)
    out[rank] = (maps, gathered, tiny_owners)
    dist.barrier()
    dist.destroy_process_group()


def test_ranks_agree_on_owners_and_reassemble_the_update():
    dmbuild.build()
    dm.lib()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, port, out)) for r in range(WORLD)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=300)
            assert p.exitcode == 0
        res = dict(out)

    from oracle import ns64

    # The owner map of the 224-matrix set: identical on both ranks, every matrix owned once, loads = the
    # summed cost of each rank's matrices.
    maps = res[0][0]
    assert maps == res[1][0]
    owners, loads = maps[0]
    assert maps[1] == (owners, loads)
    assert sorted(set(owners)) == list(range(WORLD))
    shapes = [(r, c) for _, r, c in workloads.llama3_8b_shapes(32)]
    for rank in range(WORLD):
        cost = sum(dm.gram_flops(r, c) for (r, c), o in zip(shapes, owners) if o == rank)
        assert loads[rank] == cost
    assert max(loads) / (sum(loads) / WORLD) < 1.05

    # Owned updates exchanged between ranks equal one process updating everything.
    gathered = res[0][1]
    tiny_owners = res[0][2]
    assert res[1][2] == tiny_owners
    merged = {}
    for rank, part in enumerate(gathered):
        assert all(tiny_owners[i] == rank for i in part)
        merged.update(part)
    assert sorted(merged) == list(range(len(TINY)))
    for i, s in enumerate(TINY):
        w0, g, m0 = _tiny_inputs(i, s)
        ref = ns64.muon_step(w0, g, m0, 0.02, 0.95, ns64.YOU, (2,), "gram")
        assert np.array_equal(merged[i][0], ref["W"]) and np.array_equal(merged[i][1], ref["M"])
