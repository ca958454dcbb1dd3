"""Float64 CPU oracle for the owner-rank Muon update.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference arm of ``bench.py`` may import or call this module. The CUDA library never calls it
and shares no code, table or helper with it.

What it restates (sources are web pages about DMuon / distributed Muon):

* Muon step shape -- keep a momentum M of the gradient, approximately orthogonalise M, use the
  result as the update direction: pwwt.cn "Muon 分布式技术" blog, section "2. Muon执行过程"
  (its displayed formulas were lost in extraction; the plain reading is used, see below).
* Direct Newton-Schulz, X_{k+1} = a_k X + b_k (X X^T) X + c_k (X X^T)^2 X:
  DMuon "Newton-Schulz 变体" page, section "直接空间 NS（经典）" (same equation on the DMuon
  "Core Concepts" page, section "1. Dedicated Ownership").
* Gram-space Newton-Schulz, R = X X^T, Z_k = b_k R_k + c_k R_k^2, Q_{k+1} = Z_k Q_k + a_k Q_k,
  output Q X, restart applies Q to X and recomputes R: "Newton-Schulz 变体", sections
  "Gram 空间 NS（Dao-AILab）" and "重启机制".
* Precision pipeline, X = G / (||G|| + eps) then iterate: "Newton-Schulz 变体", section "精度流水线".
  The oracle iterates in float64 throughout; the fp16 step is what the GPU path adds.
* Coefficient tables: "Newton-Schulz 变体", section "系数集" (values as printed).

Readings taken where the pages are silent (each is listed with its reason in the design notes):

* momentum is M <- beta * M + G (no (1 - beta) factor, no Nesterov term);
* the Frobenius norm of the whole momentum matrix is taken, and eps is added to the norm;
* the weight update is W <- W - lr * O with no shape factor and no weight decay;
* the Gram recurrence for R is R <- (a I + Z) R (a I + Z), which is exactly X_{k+1} X_{k+1}^T;
* a restart at index k happens before step k (default [2]: after steps 0 and 1); index 0 is a no-op;
* matrices with more rows than columns are transposed so the Gram matrix is the smaller one,
  and the output is transposed back.
"""

from __future__ import annotations

import numpy as np

# "Newton-Schulz 变体" page, section "系数集": POLAR_EXPRESS_COEFFICIENTS, printed approximations
# after the 1.05 safety factor. Used verbatim.
POLAR_EXPRESS = (
    (7.893, -20.381, 14.939),
    (3.912, -2.544, 0.470),
    (3.761, -2.512, 0.476),
    (3.160, -2.148, 0.440),
    (2.191, -1.441, 0.361),
)

# Same section: YOU_COEFFICIENTS (attributed to @YouJiacheng). Used verbatim.
YOU = (
    (4.0848, -6.8946, 2.9270),
    (3.9505, -6.3029, 2.6377),
    (3.7418, -5.5913, 2.3037),
    (2.8769, -3.1427, 1.2046),
    (2.8366, -3.0525, 1.2012),
)

# "Newton-Schulz 变体", section "重启机制": default restart list [2].
DEFAULT_RESTARTS = (2,)


def momentum(m0, g, beta):
    """M <- beta * M0 + G, in float64 (pwwt.cn blog, section 2: momentum of the gradient)."""
    return beta * np.asarray(m0, dtype=np.float64) + np.asarray(g, dtype=np.float64)


def frobenius_norm(m):
    """||M||_F = sqrt(sum of squares) in float64 ("精度流水线": G.norm())."""
    m = np.asarray(m, dtype=np.float64)
    return float(np.sqrt(np.sum(m * m)))


def normalise(m, eps):
    """X = M / (||M||_F + eps) ("精度流水线", stage 1). Returns (X, ||M||_F)."""
    m = np.asarray(m, dtype=np.float64)
    s = frobenius_norm(m)
    return m / (s + eps), s


def orient(x):
    """Put the smaller dimension first so X X^T is the small Gram matrix
    ("Gram 空间 NS": the (m, m) intermediate is smaller when m < n). Returns (X', transposed?)."""
    if x.shape[0] > x.shape[1]:
        return x.T, True
    return x, False


def ns_direct(x, coeffs):
    """Direct-space NS ("直接空间 NS"): X <- a X + b (X X^T) X + c (X X^T)^2 X for each (a, b, c)."""
    x = np.array(x, dtype=np.float64)
    for a, b, c in coeffs:
        gram = x @ x.T
        x = a * x + b * (gram @ x) + c * ((gram @ gram) @ x)
    return x


def _gram_update(r, z, a):
    """R_{k+1} from R_k and Z_k: (a I + Z) R (a I + Z) ("Gram 空间 NS": R evolves from R_k, Z_k)."""
    w = a * np.eye(r.shape[0]) + z
    return w @ r @ w


def ns_gram(x, coeffs, restarts=DEFAULT_RESTARTS):
    """Gram-space NS ("Gram 空间 NS" + "重启机制").

    R = X X^T, Q = I. For each step k: if k is a restart index (k > 0), X <- Q X, R <- X X^T, Q <- I.
    Then Z = b R + c R^2, Q <- Z Q + a Q, R <- (a I + Z) R (a I + Z). Output Q X.
    """
    x = np.array(x, dtype=np.float64)
    eye = np.eye(x.shape[0])
    r = x @ x.T
    q = eye.copy()
    restart_set = set(int(k) for k in restarts)
    for k, (a, b, c) in enumerate(coeffs):
        if k in restart_set and k > 0:
            x = q @ x
            r = x @ x.T
            q = eye.copy()
        z = b * r + c * (r @ r)
        q = z @ q + a * q
        r = _gram_update(r, z, a)
    return q @ x


def newton_schulz(g, coeffs=POLAR_EXPRESS, restarts=DEFAULT_RESTARTS, backend="gram", eps=1e-7):
    """Normalise, orient, iterate, restore orientation. Returns O with the shape of g."""
    x, _ = normalise(g, eps)
    x, transposed = orient(x)
    if backend == "gram":
        o = ns_gram(x, coeffs, restarts)
    elif backend == "direct":
        o = ns_direct(x, coeffs)
    else:
        raise ValueError(f"unknown backend {backend!r}")
    return o.T if transposed else o


def muon_step(w0, g, m0, lr, beta, coeffs=POLAR_EXPRESS, restarts=DEFAULT_RESTARTS,
              backend="gram", eps=1e-7):
    """One owner-rank Muon update of one matrix, all in float64.

    Returns a dict with the new momentum M, its Frobenius norm, the normalised and oriented X
    (before iteration), the orthogonalised O (shape of W) and the new weight W = W0 - lr * O.
    """
    m = momentum(m0, g, beta)
    x, s = normalise(m, eps)
    x_oriented, transposed = orient(x)
    if backend == "gram":
        o = ns_gram(x_oriented, coeffs, restarts)
    elif backend == "direct":
        o = ns_direct(x_oriented, coeffs)
    else:
        raise ValueError(f"unknown backend {backend!r}")
    if transposed:
        o = o.T
    w = np.asarray(w0, dtype=np.float64) - lr * o
    return {"M": m, "norm": s, "X": x_oriented, "O": o, "W": w}


def gram_by_shards(x, bounds):
    """Sum over column shards [bounds[t], bounds[t+1]) of X_t X_t^T ("Gram 空间 NS": the Gram matrix is a
    sum of local Gram matrices, which is what makes tensor parallelism exact with one all-reduce)."""
    x = np.asarray(x, dtype=np.float64)
    r = np.zeros((x.shape[0], x.shape[0]))
    for t in range(len(bounds) - 1):
        xt = x[:, bounds[t]:bounds[t + 1]]
        r += xt @ xt.T
    return r


def ns_gram_tp(x, coeffs, restarts, bounds):
    """ns_gram with every Gram formation (the first and each restart's) taken as gram_by_shards."""
    x = np.array(x, dtype=np.float64)
    eye = np.eye(x.shape[0])
    r = gram_by_shards(x, bounds)
    q = eye.copy()
    restart_set = set(int(k) for k in restarts)
    for k, (a, b, c) in enumerate(coeffs):
        if k in restart_set and k > 0:
            x = q @ x
            r = gram_by_shards(x, bounds)
            q = eye.copy()
        z = b * r + c * (r @ r)
        q = z @ q + a * q
        r = _gram_update(r, z, a)
    return q @ x


def newton_schulz_tp(g, coeffs, restarts, bounds, eps=1e-7):
    """Gram NS of g split into column shards of its long side: the squared norm is the sum of per-shard
    sums of squares, the Gram matrices sums of per-shard products. Returns O with the shape of g."""
    x, transposed = orient(np.asarray(g, dtype=np.float64))
    sumsq = sum(float(np.sum(x[:, bounds[t]:bounds[t + 1]] ** 2)) for t in range(len(bounds) - 1))
    x = x / (np.sqrt(sumsq) + eps)
    o = ns_gram_tp(x, coeffs, restarts, bounds)
    return o.T if transposed else o
