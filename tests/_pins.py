"""Helpers for the oracle pins: golden tables and the closed form of Newton-Schulz.

The closed form is the independent route: for X = U diag(s) V^T, every NS step is an odd matrix
polynomial of X, so the output is U diag(f(s')) V^T with s' = s / (||s||_2 + eps) and
f = p_5 o ... o p_1, p_k(x) = a_k x + b_k x^3 + c_k x^5 evaluated one singular value at a time.
"""

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden_coefficients():
    """Both coefficient tables from tests/golden/coefficients.txt, as tuples of float triples."""
    tables, cur = {}, None
    with open(os.path.join(GOLDEN, "coefficients.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                cur = line.strip("[]")
                tables[cur] = []
                continue
            tables[cur].append(tuple(float(v) for v in line.split()))
    return {k: tuple(v) for k, v in tables.items()}


def scalar_map(x, coeffs):
    """f(x) = p_K(...p_1(x)) for one scalar x, plain Python floats."""
    for a, b, c in coeffs:
        x = a * x + b * x ** 3 + c * x ** 5
    return x


def random_orthogonal(rng, n, k=None):
    """n x k matrix with orthonormal columns: QR of a Gaussian, signs fixed by diag(R)."""
    k = n if k is None else k
    q, r = np.linalg.qr(rng.standard_normal((n, k)))
    return q * np.sign(np.diag(r))


def closed_form(u, s, v, coeffs, eps):
    """U diag(f(s / (||s|| + eps))) V^T for X = U diag(s) V^T (columns of U, V orthonormal)."""
    sn = np.asarray(s, dtype=np.float64) / (np.sqrt(np.sum(np.square(s, dtype=np.float64))) + eps)
    fs = np.array([scalar_map(float(t), coeffs) for t in sn])
    return (u * fs) @ v.T


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))
