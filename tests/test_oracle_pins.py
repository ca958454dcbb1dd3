"""Pins for the CPU oracle: nothing here compares the oracle with itself.

Each test ties the oracle to something fixed independently of it: the tables printed on the pages
(tests/golden), the closed form U f(S) V^T of an odd matrix polynomial, exact rational arithmetic,
an SVD brute force, textbook special cases and exact invariances. The last test plants mistakes
in a copy of the oracle and checks that these pins catch every one.
"""

import inspect
import types

import numpy as np
import pytest

from oracle import exact, ns64
from tests import _pins

EPS = 1e-7


def test_coefficient_tables_match_pages():
    g = _pins.golden_coefficients()
    assert ns64.POLAR_EXPRESS == g["POLAR_EXPRESS"]
    assert ns64.YOU == g["YOU"]
    assert ns64.DEFAULT_RESTARTS == (2,)


def _spectral_case(rng, m, n, sigma):
    k = min(m, n)
    u = _pins.random_orthogonal(rng, m, k)
    v = _pins.random_orthogonal(rng, n, k)
    return (u * sigma) @ v.T, u, v


@pytest.mark.parametrize("backend", ["direct", "gram"])
@pytest.mark.parametrize("table", ["YOU", "POLAR_EXPRESS"])
@pytest.mark.parametrize("shape", [(48, 80), (80, 48), (64, 64), (1, 7)])
def test_closed_form_log_uniform(backend, table, shape):
    """X = U S V^T with log-uniform S in [1e-6, 1] (the closed-form workload, scaled down)."""
    rng = np.random.default_rng(11)
    m, n = shape
    k = min(m, n)
    sigma = 10.0 ** rng.uniform(-6.0, 0.0, size=k)
    x, u, v = _spectral_case(rng, m, n, sigma)
    coeffs = getattr(ns64, table)
    got = ns64.newton_schulz(x, coeffs, (2,), backend, EPS)
    want = _pins.closed_form(u, sigma, v, coeffs, EPS)
    assert _pins.rel_fro(got, want) < 1e-10


@pytest.mark.parametrize("backend", ["direct", "gram"])
def test_closed_form_top_tenth(backend):
    """Top 10% of singular values at 1, the rest at 1e-4 (the second closed-form workload, scaled)."""
    rng = np.random.default_rng(12)
    m, n = 100, 400
    sigma = np.full(m, 1e-4)
    sigma[: round(0.1 * m)] = 1.0
    x, u, v = _spectral_case(rng, m, n, sigma)
    got = ns64.newton_schulz(x, ns64.POLAR_EXPRESS, (2,), backend, EPS)
    want = _pins.closed_form(u, sigma, v, ns64.POLAR_EXPRESS, EPS)
    assert _pins.rel_fro(got, want) < 1e-10


@pytest.mark.parametrize("restarts", [(2,), (1, 3), (), (1, 2, 3, 4), (0,)])
def test_exact_gram_equals_direct(restarts):
    """In exact arithmetic Gram NS with any restart list is the direct iteration."""
    rng = np.random.default_rng(13)
    x, _ = ns64.normalise(rng.standard_normal((4, 8)), EPS)
    xe = exact.from_floats(x.tolist())
    d = exact.ns_direct(xe, ns64.YOU)
    g = exact.ns_gram(xe, ns64.YOU, restarts)
    assert exact.equal(d, g)


def test_fp64_oracle_matches_exact():
    rng = np.random.default_rng(14)
    for table in (ns64.YOU, ns64.POLAR_EXPRESS):
        x, _ = ns64.normalise(rng.standard_normal((3, 7)) * 0.3, EPS)
        xe = exact.from_floats(x.tolist())
        want = np.array(exact.to_floats(exact.ns_direct(xe, table)))
        assert np.abs(ns64.ns_direct(x, table) - want).max() < 1e-12 * max(1.0, np.abs(want).max())
        assert np.abs(ns64.ns_gram(x, table, (2,)) - want).max() < 1e-12 * max(1.0, np.abs(want).max())


@pytest.mark.parametrize("shape", [(4, 8), (8, 4), (16, 16), (5, 33)])
def test_svd_brute_force(shape):
    """numpy's SVD gives U S V^T; the output must be U f(S') V^T."""
    rng = np.random.default_rng(15)
    g = rng.standard_normal(shape)
    u, s, vt = np.linalg.svd(g, full_matrices=False)
    want = _pins.closed_form(u, s, vt.T, ns64.YOU, EPS)
    for backend in ("direct", "gram"):
        assert _pins.rel_fro(ns64.newton_schulz(g, ns64.YOU, (2,), backend, EPS), want) < 1e-11


def test_zero_steps_and_identity_polynomial_return_x():
    rng = np.random.default_rng(16)
    x, _ = ns64.normalise(rng.standard_normal((6, 10)), EPS)
    assert np.array_equal(ns64.ns_direct(x, ()), x)
    assert np.allclose(ns64.ns_gram(x, (), (2,)), x, atol=0, rtol=0)
    ident = ((1.0, 0.0, 0.0),) * 5
    assert np.allclose(ns64.ns_direct(x, ident), x, rtol=0, atol=1e-15)
    assert np.allclose(ns64.ns_gram(x, ident, (2,)), x, rtol=0, atol=1e-15)


def test_classic_cubic_one_step():
    """(a, b, c) = (1.5, -0.5, 0): one step maps each singular value s to 1.5 s - 0.5 s^3."""
    rng = np.random.default_rng(17)
    sigma = np.array([0.9, 0.5, 0.1])
    x, u, v = _spectral_case(rng, 3, 5, sigma)
    for fn in (lambda z: ns64.ns_direct(z, ((1.5, -0.5, 0.0),)),
               lambda z: ns64.ns_gram(z, ((1.5, -0.5, 0.0),), ())):
        assert np.allclose(fn(x), (u * (1.5 * sigma - 0.5 * sigma ** 3)) @ v.T, rtol=0, atol=1e-15)


def test_zero_gradient_gives_zero_update():
    z = np.zeros((5, 9))
    for backend in ("direct", "gram"):
        assert not np.any(ns64.newton_schulz(z, ns64.POLAR_EXPRESS, (2,), backend, EPS))
    out = ns64.muon_step(np.ones((5, 9)), z, z, 0.02, 0.95, ns64.YOU, (2,), "gram", EPS)
    assert np.array_equal(out["W"], np.ones((5, 9))) and out["norm"] == 0.0


def test_orthonormal_rows():
    """Orthonormal rows: every normalised singular value is 1/sqrt(m) (up to eps)."""
    rng = np.random.default_rng(18)
    m, n = 8, 24
    g = _pins.random_orthogonal(rng, n, m).T
    s = 1.0 / (np.sqrt(m) + EPS)
    want = _pins.scalar_map(s, ns64.YOU) * g
    for backend in ("direct", "gram"):
        assert np.allclose(ns64.newton_schulz(g, ns64.YOU, (2,), backend, EPS), want, rtol=0, atol=1e-13)


def test_single_row():
    """m = 1: R is the 1x1 scalar |x|^2 and the map is f applied to |x|."""
    g = np.array([[3.0, 4.0]])
    want = _pins.scalar_map(5.0 / (5.0 + EPS), ns64.YOU) * g / 5.0
    for backend in ("direct", "gram"):
        assert np.allclose(ns64.newton_schulz(g, ns64.YOU, (2,), backend, EPS), want, rtol=1e-14, atol=0)


@pytest.mark.parametrize("backend", ["direct", "gram"])
def test_invariances(backend):
    rng = np.random.default_rng(19)
    g = rng.standard_normal((12, 20))
    ns = lambda z: ns64.newton_schulz(z, ns64.YOU, (2,), backend, EPS)  # noqa: E731
    o = ns(g)
    assert np.allclose(ns(g.T), o.T, rtol=0, atol=1e-12)
    assert np.allclose(ns(-g), -o, rtol=0, atol=1e-12)
    assert np.allclose(ns(7.5 * g), o, rtol=0, atol=1e-6)  # scale-invariant up to eps
    u = _pins.random_orthogonal(rng, 12)
    v = _pins.random_orthogonal(rng, 20)
    assert np.allclose(ns(u @ g @ v), u @ o @ v, rtol=0, atol=1e-12)


def test_restart_lists_agree_in_float64():
    rng = np.random.default_rng(20)
    x, _ = ns64.normalise(rng.standard_normal((30, 50)), EPS)
    base = ns64.ns_direct(x, ns64.POLAR_EXPRESS)
    for rs in ((2,), (1, 3), (), (1, 2, 3, 4)):
        assert _pins.rel_fro(ns64.ns_gram(x, ns64.POLAR_EXPRESS, rs), base) < 1e-11


def test_momentum_and_norm_small_exact():
    m0 = np.array([[1.0, 2.0], [0.0, -4.0]])
    g = np.array([[3.0, 4.0], [1.0, 0.5]])
    m = ns64.momentum(m0, g, 0.5)
    assert np.array_equal(m, [[3.5, 5.0], [1.0, -1.5]])
    assert ns64.frobenius_norm(m) == np.sqrt(3.5 ** 2 + 25.0 + 1.0 + 2.25)
    x, s = ns64.normalise(m, 0.25)
    assert np.array_equal(x, m / (s + 0.25))


def test_muon_step_composition():
    rng = np.random.default_rng(21)
    w0 = rng.standard_normal((9, 4))
    g = rng.standard_normal((9, 4))
    m0 = rng.standard_normal((9, 4))
    out = ns64.muon_step(w0, g, m0, 0.02, 0.95, ns64.YOU, (2,), "gram", EPS)
    assert out["X"].shape == (4, 9)  # tall input is worked on transposed
    m = 0.95 * m0 + g
    u, s, vt = np.linalg.svd(m, full_matrices=False)
    o = _pins.closed_form(u, s, vt.T, ns64.YOU, EPS)
    assert np.allclose(out["M"], m, rtol=0, atol=0)
    assert _pins.rel_fro(out["O"], o) < 1e-11
    assert np.allclose(out["W"], w0 - 0.02 * out["O"], rtol=0, atol=1e-15)


# --- planted mistakes ---------------------------------------------------------------------------
# Not in the list: skipping the recomputation of R at a restart. In exact arithmetic the recurrence
# already gives R = X X^T there, so that change alters rounding only and no exact pin can see it.

MUTATIONS = [
    ("x = a * x + b * (gram @ x) + c * ((gram @ gram) @ x)", "x = a * x + b * (gram @ x) + c * (gram @ x)"),
    ("gram = x @ x.T", "gram = x.T @ x"),
    ("q = z @ q + a * q", "q = z @ q - a * q"),
    ("return w @ r @ w", "return w @ r"),
    ("w = a * np.eye(r.shape[0]) + z", "w = z"),
    ("            x = q @ x\n", "            x = x\n"),
    ("z = b * r + c * (r @ r)", "z = c * r + b * (r @ r)"),
    ("return m / (s + eps), s", "return m / (s * s + eps), s"),
    ("return beta * np.asarray(m0, dtype=np.float64) + np.asarray(g, dtype=np.float64)",
     "return beta * np.asarray(m0, dtype=np.float64) + (1 - beta) * np.asarray(g, dtype=np.float64)"),
    ("return o.T if transposed else o", "return o"),
]


def _mutant(old, new):
    src = inspect.getsource(ns64)
    assert src.count(old) >= 1, old
    mod = types.ModuleType("ns64_mutant")
    exec(compile(src.replace(old, new), "ns64_mutant", "exec"), mod.__dict__)
    return mod


def _pins_pass(mod):
    """The pins above, run against a given module; False as soon as one fails."""
    try:
        rng = np.random.default_rng(31)
        for m, n in ((6, 10), (10, 6), (7, 7)):
            k = min(m, n)
            sigma = 10.0 ** rng.uniform(-3.0, 0.0, size=k)
            x, u, v = _spectral_case(rng, m, n, sigma)
            want = _pins.closed_form(u, sigma, v, mod.YOU, EPS)
            for backend in ("direct", "gram"):
                if _pins.rel_fro(mod.newton_schulz(x, mod.YOU, (2,), backend, EPS), want) > 1e-10:
                    return False
        m0 = np.array([[1.0, 2.0], [0.0, -4.0]])
        g = np.array([[3.0, 4.0], [1.0, 0.5]])
        if not np.array_equal(mod.momentum(m0, g, 0.5), [[3.5, 5.0], [1.0, -1.5]]):
            return False
        return True
    except Exception:
        return False


def test_pins_pass_on_the_oracle():
    assert _pins_pass(ns64)


@pytest.mark.parametrize("old,new", MUTATIONS, ids=[f"m{i}" for i in range(len(MUTATIONS))])
def test_pins_catch_planted_mistake(old, new):
    assert not _pins_pass(_mutant(old, new))
