"""Pins for the AdamW oracle: PyTorch's own AdamW in float64 (a library routine), closed forms of the
first step and of a constant gradient, pure weight decay, and planted mistakes that must be caught."""

import inspect
import types

import numpy as np
import torch

from oracle import adamw

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _run(mod, p, gs, m=None, v=None):
    m = np.zeros_like(p) if m is None else m
    v = np.zeros_like(p) if v is None else v
    for t, g in enumerate(gs, start=1):
        p, m, v = mod.adamw_step(p, g, m, v, HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], HP["weight_decay"], t)
    return p, m, v


def _torch_adamw(p0, gs):
    p = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.AdamW([p], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            weight_decay=HP["weight_decay"])
    for g in gs:
        p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
    st = opt.state[p]
    return p.detach().numpy(), st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()


def _pins_pass(mod):
    rng = np.random.default_rng(3)
    p0 = rng.standard_normal(257) * 0.02
    gs = [rng.standard_normal(257) * 1e-3 for _ in range(4)]
    try:
        got = _run(mod, p0.copy(), gs)
        want = _torch_adamw(p0.copy(), gs)
        if not all(np.allclose(a, b, rtol=1e-12, atol=1e-15) for a, b in zip(got, want)):
            return False
        # first step from zero state: p1 = p0 (1 - lr wd) - lr g / (|g| + eps)
        p1, _, _ = _run(mod, p0.copy(), gs[:1])
        closed = p0 * (1 - HP["lr"] * HP["weight_decay"]) - HP["lr"] * gs[0] / (np.abs(gs[0]) + HP["eps"])
        if not np.allclose(p1, closed, rtol=1e-12, atol=1e-15):
            return False
        # zero gradient: pure decoupled decay
        pz, _, _ = _run(mod, p0.copy(), [np.zeros(257)] * 3)
        if not np.allclose(pz, p0 * (1 - HP["lr"] * HP["weight_decay"]) ** 3, rtol=1e-14, atol=0):
            return False
        return True
    except Exception:
        return False


def test_oracle_passes_pins():
    assert _pins_pass(adamw)


def test_constant_gradient_closed_form():
    """With the same gradient every step the bias-corrected moments are exactly g and g^2."""
    p0 = np.array([0.5, -0.25, 0.0, 1.0])
    g = np.array([1e-3, -2e-3, 5e-4, 0.0])
    p, _, _ = _run(adamw, p0.copy(), [g] * 5)
    want = p0.copy()
    for _ in range(5):
        want = want * (1 - HP["lr"] * HP["weight_decay"]) - HP["lr"] * g / (np.abs(g) + HP["eps"])
    assert np.allclose(p, want, rtol=1e-12, atol=1e-15)


MUTATIONS = [
    ("bc1 = 1.0 - beta1 ** step", "bc1 = 1.0"),
    ("bc2 = 1.0 - beta2 ** step", "bc2 = 1.0"),
    ("* (1.0 - lr * weight_decay)", "* 1.0"),
    ("(1.0 - beta2) * g * g", "(1.0 - beta2) * g"),
    ("np.sqrt(v) / np.sqrt(bc2) + eps", "np.sqrt(v / bc2 + eps)"),
]


def test_pins_catch_planted_mistakes():
    src = inspect.getsource(adamw)
    for old, new in MUTATIONS:
        assert old in src, old
        mod = types.ModuleType("adamw_mutant")
        exec(compile(src.replace(old, new), "adamw_mutant", "exec"), mod.__dict__)
        assert not _pins_pass(mod), old
