"""Pins for the fp16 error model (oracle/fp16_model.py), which predicts the error floor of an fp16 iteration.

With float64 storage the model rounds nothing, so it must give the closed form U f(S) V^T of the odd matrix
polynomial, like the oracle; mistakes planted in a copy of it must break that. With fp16 storage it must round
what it stores and land at a plausible fp16 error.
"""

import inspect
import types

import numpy as np
import pytest

from oracle import fp16_model
from tests import _pins

EPS = 1e-7
TABLES = _pins.golden_coefficients()


def _spectral(rng, m, n, sigma):
    k = min(m, n)
    u = _pins.random_orthogonal(rng, m, k)
    v = _pins.random_orthogonal(rng, n, k)
    return (u * sigma) @ v.T, u, v


def _closed_form_holds(mod, tol=1e-10):
    rng = np.random.default_rng(41)
    for m, n in ((6, 10), (10, 6), (7, 7), (1, 5)):
        k = min(m, n)
        sigma = 10.0 ** rng.uniform(-3.0, 0.0, size=k)
        x, u, v = _spectral(rng, m, n, sigma)
        for name in ("YOU", "POLAR_EXPRESS"):
            want = _pins.closed_form(u, sigma, v, TABLES[name], EPS)
            for backend, restarts in (("direct", (2,)), ("gram", (2,)), ("gram", ()), ("gram", (1, 3)),
                                      ("gram", (1, 2, 3, 4))):
                got = mod.newton_schulz(x, TABLES[name], restarts, backend, EPS, store=np.float64)
                if _pins.rel_fro(got, want) > tol:
                    return False
    return True


def test_float64_storage_gives_the_closed_form():
    assert _closed_form_holds(fp16_model)


MUTATIONS = [
    ("nxt = p.mm(poly, x) + a * x", "nxt = p.mm(poly, x)"),
    ("poly = p.keep(c * p.mm(gram, gram) + b * gram)", "poly = p.keep(b * p.mm(gram, gram) + c * gram)"),
    ("gram = p.keep(p.mm(x, x.T))", "gram = p.keep(p.mm(x.T, x))"),
    ("zv = c * p.mm(r, r) + b * r", "zv = c * p.mm(r, r) - b * r"),
    ("q = p.keep(zv + a * eye) if q is None", "q = p.keep(zv) if q is None"),
    ("else p.keep(p.mm(z, q) + a * q)", "else p.keep(p.mm(q, z))"),
    ("s = p.keep(p.mm(z, r) + a * r)", "s = p.keep(p.mm(z, r))"),
    ("r = p.keep(p.mm(s, z) + a * s)", "r = p.keep(p.mm(s, z) + a * r)"),
    ("            x = p.keep(p.mm(q, x))\n", "            x = p.keep(x)\n"),
    ("inv = p.acc(1.0 / (s + eps))", "inv = p.acc(1.0 / (s * s + eps))"),
    ("o = o.T if transposed else o", "o = o"),
]


def _mutant(old, new):
    src = inspect.getsource(fp16_model)
    assert src.count(old) == 1, old
    mod = types.ModuleType("fp16_model_mutant")
    exec(compile(src.replace(old, new), "fp16_model_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("old,new", MUTATIONS, ids=[f"m{i}" for i in range(len(MUTATIONS))])
def test_closed_form_catches_planted_mistake(old, new):
    try:
        with np.errstate(all="ignore"):
            ok = _closed_form_holds(_mutant(old, new))
    except Exception:
        ok = False
    assert not ok


def test_fp16_storage_rounds_what_it_stores():
    rng = np.random.default_rng(42)
    g = rng.standard_normal((40, 90)).astype(np.float32)
    x, transposed = fp16_model.x_from_momentum(g, EPS)
    assert not transposed and x.dtype == np.float32
    assert np.array_equal(x.astype(np.float16).astype(np.float32), x)
    # one fp16 rounding of X: relative error at most 2^-11 per element in fp16's normal range (the fp32
    # product before it adds ~1e-7), absolute error at most 2^-25 below it
    exact = g.astype(np.float64) / (np.linalg.norm(g.astype(np.float64)) + EPS)
    normal = np.abs(exact) >= 2.0 ** -14
    assert np.max(np.abs(x - exact)[normal] / np.abs(exact)[normal]) <= 2.0 ** -11 * 1.01
    assert np.max(np.abs(x - exact)[~normal], initial=0.0) <= 2.0 ** -25 * 1.01
    xt, tt = fp16_model.x_from_momentum(g.T, EPS)
    assert tt and np.array_equal(xt, x)


@pytest.mark.parametrize("backend", ["direct", "gram"])
def test_fp16_error_is_an_fp16_error(backend):
    """YOU on a 128 x 512 Gaussian: the fp16 model lies well off float64 accuracy and well inside 2e-2."""
    rng = np.random.default_rng(43)
    g = rng.standard_normal((128, 512))
    u, s, vt = np.linalg.svd(g, full_matrices=False)
    want = _pins.closed_form(u, s, vt.T, TABLES["YOU"], EPS)
    err = _pins.rel_fro(fp16_model.newton_schulz(g, TABLES["YOU"], (2,), backend, EPS), want)
    assert 1e-4 < err < 1e-2, err



def test_floor_separates_transposed_operands():
    """The GPU floor test's upper bound (1.5 times the floor) sees a real mistake: reading the second operand
    of R^2, Z R and S Z transposed (the same product in exact arithmetic, where R, Z and S are symmetric, but
    not for their fp16-stored values) lifts the 256 x 1024 Gram error to about 2.2 times the floor."""
    rng = np.random.default_rng(44)
    g = rng.standard_normal((256, 1024)).astype(np.float32)
    u, s, vt = np.linalg.svd(g.astype(np.float64), full_matrices=False)
    want = _pins.closed_form(u, s, vt.T, TABLES["YOU"], EPS)
    floor = _pins.rel_fro(fp16_model.newton_schulz(g, TABLES["YOU"], (2,), "gram", EPS), want)
    src = inspect.getsource(fp16_model)
    for old, new in (("zv = c * p.mm(r, r) + b * r", "zv = c * p.mm(r, r.T) + b * r"),
                     ("s = p.keep(p.mm(z, r) + a * r)", "s = p.keep(p.mm(z, r.T) + a * r)"),
                     ("r = p.keep(p.mm(s, z) + a * s)", "r = p.keep(p.mm(s, z.T) + a * s)")):
        assert src.count(old) == 1, old
        src = src.replace(old, new)
    mod = types.ModuleType("fp16_model_transposed")
    exec(compile(src, "fp16_model_transposed", "exec"), mod.__dict__)
    err = _pins.rel_fro(mod.newton_schulz(g, TABLES["YOU"], (2,), "gram", EPS), want)
    assert 5e-4 < floor < 2e-3
    assert err > 1.8 * floor, (floor, err)
