"""fp16 error model of the Newton-Schulz iteration: what an fp16 implementation can reach at best.

TEST INFRASTRUCTURE, and NOT an oracle. Only ``tests/`` may import it. It shares no code with the CUDA
library (nor with ``ns64``, so that reducing it to float64 checks it against the oracle independently).

The pages fix the precision pipeline only as "fp32 normalisation, then fp16 iteration" ("Newton-Schulz 变体",
section "精度流水线"). This module plays the iteration through with the precisions the library uses at each
stage, in NumPy:

* X = fp16(M * inv), with M in fp32 and inv = fp32(1 / (||M||_F + eps)) from a float64 norm;
* every product has fp16 operands and fp32 accumulation (NumPy float32 matmul of fp16-rounded values:
  the summation order differs from a tensor core's, the precision does not);
* each step's scalar recipe runs in fp32 on the fp32 product, and the result is stored as fp16 (round to
  nearest even) -- R, Z, Q, S and X between phases;
* the output Q X (or B X + a X) stays fp32.

The iteration follows the same steps as the oracle (direct: X X^T, B = b A + c A^2, B X + a X; Gram: R = X X^T,
Z = b R + c R^2, Q = Z + a I after a (re)start and Z Q + a Q otherwise, R <- (aI + Z) R (aI + Z) as
S = Z R + a R then S Z + a S when the next step uses it, restart X <- Q X, R <- X X^T), so its distance from
the float64 oracle is the error that fp16 storage alone causes. The GPU's error against the oracle can then be
judged against this floor: a kernel that is as accurate as fp16 allows lands near it.

With ``store=np.float64`` nothing is rounded and products accumulate in float64: the model must then agree
with the oracle to rounding (the pin in ``tests/test_fp16_model.py``, which also plants mistakes in a copy of this module).
"""

from __future__ import annotations

import numpy as np


class _Precision:
    """Rounding of stored values and accumulation type of products."""

    def __init__(self, store):
        self.store = np.dtype(store)
        self.acc = np.float64 if self.store == np.float64 else np.float32

    def keep(self, v):
        """v (an accumulator-precision array) stored and read back."""
        return np.asarray(v).astype(self.store).astype(self.acc)

    def mm(self, a, b):
        return np.asarray(a, dtype=self.acc) @ np.asarray(b, dtype=self.acc)


def x_from_momentum(m, eps, store=np.float16):
    """X = store(M * inv) with inv = fp32(1 / (||M||_F + eps)), the norm summed in float64 (fp32 M in the
    fp16 model). Returns (X oriented so rows <= cols, transposed?)."""
    p = _Precision(store)
    m = np.asarray(m, dtype=p.acc)
    s = float(np.sqrt(np.sum(m.astype(np.float64) ** 2)))
    inv = p.acc(1.0 / (s + eps))
    x = p.keep(m * inv)
    if x.shape[0] > x.shape[1]:
        return x.T.copy(), True
    return x, False


def direct(x, coeffs, store=np.float16):
    """Direct iteration with stored intermediates: A = X X^T, B = b A + c A^2, X <- B X + a X; the last X in
    accumulator precision."""
    p = _Precision(store)
    x = p.keep(x)
    for k, (a, b, c) in enumerate(coeffs):
        gram = p.keep(p.mm(x, x.T))
        poly = p.keep(c * p.mm(gram, gram) + b * gram)
        nxt = p.mm(poly, x) + a * x
        x = nxt if k + 1 == len(coeffs) else p.keep(nxt)
    return x


def gram(x, coeffs, restarts=(2,), store=np.float16):
    """Gram iteration with stored intermediates; returns Q X in accumulator precision."""
    p = _Precision(store)
    x = p.keep(x)
    m = x.shape[0]
    eye = np.eye(m, dtype=p.acc)
    steps = len(coeffs)
    rs = {int(k) for k in restarts if 0 < int(k) < steps}
    r = p.keep(p.mm(x, x.T))
    q = None  # identity until the first step after a (re)start
    for k, (a, b, c) in enumerate(coeffs):
        if k in rs:
            x = p.keep(p.mm(q, x))
            r = p.keep(p.mm(x, x.T))
            q = None
        zv = c * p.mm(r, r) + b * r
        z = p.keep(zv)
        q = p.keep(zv + a * eye) if q is None else p.keep(p.mm(z, q) + a * q)
        if k + 1 < steps and (k + 1) not in rs:
            s = p.keep(p.mm(z, r) + a * r)
            r = p.keep(p.mm(s, z) + a * s)
    return p.mm(q, x)


def newton_schulz(g, coeffs, restarts=(2,), backend="gram", eps=1e-7, store=np.float16):
    """The model's output O for a gradient (or momentum) g, in g's orientation, as float64."""
    x, transposed = x_from_momentum(g, eps, store)
    o = gram(x, coeffs, restarts, store) if backend == "gram" else direct(x, coeffs, store)
    o = o.T if transposed else o
    return np.asarray(o, dtype=np.float64)
