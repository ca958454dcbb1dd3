"""Dedicated ownership (LPT): the library against the oracle's plain restatement, bit-exact on the
assignment (integer work), with the oracle pinned by brute-force optima and Graham's LPT bound."""

import random

import pytest

import newton_schulz_momentum_gb300 as dm
import workloads
from newton_schulz_momentum_gb300 import build as dmbuild
from oracle import partition


@pytest.fixture(scope="module")
def lib_ready():
    dmbuild.build()
    dm.lib()


def _random_instance(rng, n, with_layers):
    shapes = [(rng.choice([128, 512, 1024, 4096, 14336]), rng.choice([128, 512, 1024, 4096, 14336])) for _ in range(n)]
    layers = [rng.randrange(max(1, n // 5)) for _ in range(n)] if with_layers else None
    return shapes, layers


@pytest.mark.parametrize("model", ["elements", "gram_flops", "direct_flops"])
@pytest.mark.parametrize("with_layers", [False, True])
def test_library_matches_oracle_exactly(lib_ready, model, with_layers):
    rng = random.Random(hash((model, with_layers)) & 0xFFFF)
    for trial in range(25):
        n = rng.randrange(1, 60)
        nranks = rng.randrange(1, 17)
        shapes, layers = _random_instance(rng, n, with_layers)
        got, loads = dm.assign_owners(shapes, nranks, layers, model)
        costs = [partition.cost(r, c, model) for r, c in shapes]
        want, want_loads = partition.lpt_assign(costs, nranks, layers)
        assert got == want
        assert loads == pytest.approx(want_loads, rel=1e-12)


def test_oracle_lpt_within_graham_bound():
    """Graham (1969): LPT makespan <= (4/3 - 1/(3R)) OPT; brute-force OPT on tiny instances."""
    rng = random.Random(5)
    for _ in range(60):
        n = rng.randrange(2, 8)
        nranks = rng.randrange(2, 4)
        costs = [float(rng.randrange(1, 20)) for _ in range(n)]
        _, load = partition.lpt_assign(costs, nranks)
        opt = partition.optimal_makespan(costs, nranks)
        assert max(load) <= (4.0 / 3.0 - 1.0 / (3 * nranks)) * opt + 1e-9
        assert max(load) >= opt


def test_oracle_known_lpt_worst_case():
    """The classic tight instance for R = 2: costs 3, 3, 2, 2, 2 -> LPT 7, optimum 6."""
    _, load = partition.lpt_assign([3.0, 3.0, 2.0, 2.0, 2.0], 2)
    assert max(load) == 7.0
    assert partition.optimal_makespan([3.0, 3.0, 2.0, 2.0, 2.0], 2) == 6.0


def test_layer_spread_and_balance_on_the_8b_set(lib_ready):
    shapes = workloads.llama3_8b_shapes(32)
    layers = [int(name.split(".")[1]) for name, _, _ in shapes]
    for nranks in (2, 4, 7, 8, 16):
        owners, loads = dm.assign_owners([(r, c) for _, r, c in shapes], nranks, layers, "gram_flops")
        for layer in range(32):
            counts = [0] * nranks
            for o, l in zip(owners, layers):
                if l == layer:
                    counts[o] += 1
            assert max(counts) - min(counts) <= 1  # a layer's 7 matrices as spread as the ranks allow
        assert max(loads) / (sum(loads) / nranks) < 1.1


def test_single_rank_and_invalid_arguments(lib_ready):
    owners, loads = dm.assign_owners([(4, 8), (16, 2)], 1)
    assert owners == [0, 0] and loads[0] == pytest.approx(6 * 16 * 8 + 17 * 64 + 6 * 4 * 16 + 17 * 8)
    with pytest.raises(dm.DmuonError):
        dm.assign_owners([(4, 8)], 0)
    with pytest.raises(dm.DmuonError):
        dm.assign_owners([(0, 8)], 2)
