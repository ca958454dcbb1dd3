"""Dedicated ownership by LPT, restated plainly (TEST INFRASTRUCTURE, like the rest of oracle/).

Source: DMuon "Core Concepts" page, section "均衡划分" (balanced partition): dedicate_params() uses LPT
(longest processing time first) with two aims, global balance of the per-rank work and the parameters
of one layer spread over different ranks; the "Newton-Schulz 变体" page, section "TP 路由", calls the
assignment deterministic. Reading taken: matrices in decreasing cost (ties by index); each goes to the
rank holding the fewest matrices of its layer, and among those to the least-loaded rank (ties by rank).

Also here, for pins only: the brute-force optimal makespan of tiny instances.
"""

from __future__ import annotations

import itertools


def cost(rows, cols, model):
    m, n = min(rows, cols), max(rows, cols)
    if model == "gram_flops":
        return 6.0 * m * m * n + 17.0 * m ** 3
    if model == "direct_flops":
        return 15.0 * m * m * n + 5.0 * m ** 3
    return float(rows) * float(cols)


def lpt_assign(costs, nranks, layers=None):
    """Owner rank per item and the load per rank."""
    order = sorted(range(len(costs)), key=lambda i: (-costs[i], i))
    load = [0.0] * nranks
    held = {}
    owner = [None] * len(costs)
    for i in order:
        if layers is None:
            candidates = list(range(nranks))
        else:
            counts = held.setdefault(layers[i], [0] * nranks)
            fewest = min(counts)
            candidates = [r for r in range(nranks) if counts[r] == fewest]
        best = min(candidates, key=lambda r: (load[r], r))
        owner[i] = best
        load[best] += costs[i]
        if layers is not None:
            held[layers[i]][best] += 1
    return owner, load


def optimal_makespan(costs, nranks):
    """Smallest possible maximum load, by trying every assignment (tiny inputs only)."""
    best = float("inf")
    for assign in itertools.product(range(nranks), repeat=len(costs)):
        if assign and assign[0] != 0:
            continue  # ranks are interchangeable: fix the first item on rank 0
        load = [0.0] * nranks
        for c, r in zip(costs, assign):
            load[r] += c
        best = min(best, max(load))
    return best
