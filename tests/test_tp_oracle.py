"""Pins for the tensor-parallel restatement of the Gram form: the split Gram matrix equals the whole one
exactly (rational arithmetic), and the split iteration reproduces the closed form and the unsplit one."""

import numpy as np
import pytest

from oracle import exact, ns64
from tests import _pins


def bounds_for(n, shards):
    return [(t * n // shards) // 8 * 8 for t in range(shards)] + [n]


def test_split_gram_is_exactly_the_gram():
    rng = np.random.default_rng(41)
    x = rng.standard_normal((4, 24))
    xe = exact.from_floats(x.tolist())
    whole = exact.matmul(xe, exact.transpose(xe))
    for bounds in ([0, 8, 24], [0, 8, 16, 24], [0, 24]):
        acc = None
        for t in range(len(bounds) - 1):
            shard = exact.from_floats(x[:, bounds[t]:bounds[t + 1]].tolist())
            g = exact.matmul(shard, exact.transpose(shard))
            acc = g if acc is None else exact.add(acc, g)
        assert exact.equal(acc, whole)


@pytest.mark.parametrize("shards", [1, 2, 3, 8])
@pytest.mark.parametrize("shape", [(48, 160), (160, 48)])
def test_split_iteration_matches_closed_form(shards, shape):
    rng = np.random.default_rng(42)
    m, n = shape
    k = min(m, n)
    sigma = 10.0 ** rng.uniform(-4.0, 0.0, size=k)
    u = _pins.random_orthogonal(rng, m, k)
    v = _pins.random_orthogonal(rng, n, k)
    g = (u * sigma) @ v.T
    bounds = bounds_for(max(m, n), shards)
    got = ns64.newton_schulz_tp(g, ns64.YOU, (2,), bounds, 1e-7)
    assert _pins.rel_fro(got, _pins.closed_form(u, sigma, v, ns64.YOU, 1e-7)) < 1e-10
    assert _pins.rel_fro(got, ns64.newton_schulz(g, ns64.YOU, (2,), "gram", 1e-7)) < 1e-12
