"""AdamW for the parameters that are not Muon targets, restated in float64 (TEST INFRASTRUCTURE, like the
rest of oracle/: only tests and the CPU baseline use it).

Source: DMuon "Core Concepts" page, section "1. Dedicated Ownership", step 6 of the per-step order: every
rank updates its FSDP2 shards of the non-dedicated parameters with AdamW. The pages name the optimizer
without restating it; the reading taken is AdamW with decoupled weight decay as PyTorch's AdamW applies
it, for step t (counted from 1):

    p <- p * (1 - lr * weight_decay)
    m <- beta1 * m + (1 - beta1) * g
    v <- beta2 * v + (1 - beta2) * g^2
    p <- p - (lr / (1 - beta1^t)) * m / (sqrt(v) / sqrt(1 - beta2^t) + eps)
"""

from __future__ import annotations

import numpy as np


def adamw_step(p, g, m, v, lr, beta1, beta2, eps, weight_decay, step):
    """One AdamW step in float64; returns (p, m, v)."""
    p = np.asarray(p, dtype=np.float64) * (1.0 - lr * weight_decay)
    g = np.asarray(g, dtype=np.float64)
    m = beta1 * np.asarray(m, dtype=np.float64) + (1.0 - beta1) * g
    v = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * g * g
    bc1 = 1.0 - beta1 ** step
    bc2 = 1.0 - beta2 ** step
    p = p - (lr / bc1) * m / (np.sqrt(v) / np.sqrt(bc2) + eps)
    return p, m, v
