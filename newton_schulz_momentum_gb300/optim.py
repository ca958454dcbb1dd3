"""The DMuon pages' Python surface over the C library: `newton_schulz(G, coefficients=..., restart_iterations=...)`,
`NewtonSchulz(backend, coefficients, restart_iterations)` and `Muon(model, lr, ns_backend)` ("Newton-Schulz
变体", section "使用自定义系数集"). Argument marshalling only: every step runs in libdmuon's kernels.

`Muon` is a `torch.optim.Optimizer`: the matrix parameters get the owner-rank Muon update (momentum,
Frobenius normalisation, fp16 Newton-Schulz, weight update) in one `dmuon_muon_step` call per step, and
the other parameters AdamW in one `dmuon_adamw_step` call ("Core Concepts" §1: dedicated matrices run
Muon, the rest AdamW). Parameters must be fp32 CUDA tensors (the update is written into fp32 weights).
"""

from __future__ import annotations

import torch

from . import (BACKENDS, DEFAULT_RESTARTS, POLAR_EXPRESS, AdamWStep, MuonStep, ns)


def newton_schulz(G, coefficients=POLAR_EXPRESS, restart_iterations=DEFAULT_RESTARTS, backend="gram", eps=1e-7,
                  stream=None):
    """NS(G / (||G||_F + eps)) of one 2-D CUDA matrix, returned as a new fp32 tensor (G is not modified):
    one `dmuon_ns` call on a copy."""
    if G.dim() != 2 or not G.is_cuda:
        raise ValueError("G must be a 2-D CUDA tensor")
    x = G.detach().to(torch.float32, copy=True).contiguous()
    return ns(x, coefficients, restart_iterations, backend, eps, stream)


class NewtonSchulz:
    """A reusable orthogonaliser with fixed form, coefficients and restart list: `NewtonSchulz("gram",
    POLAR_EXPRESS, (2,))(G)` is `newton_schulz(G, POLAR_EXPRESS, (2,), "gram")`."""

    def __init__(self, backend="gram", coefficients=POLAR_EXPRESS, restart_iterations=DEFAULT_RESTARTS, eps=1e-7):
        if backend not in BACKENDS:
            raise ValueError(f"backend must be one of {sorted(BACKENDS)}")
        self.backend = backend
        self.coefficients = tuple(tuple(float(v) for v in c) for c in coefficients)
        self.restart_iterations = tuple(int(r) for r in restart_iterations)
        self.eps = float(eps)

    def __call__(self, G, stream=None):
        return newton_schulz(G, self.coefficients, self.restart_iterations, self.backend, self.eps, stream)


def default_muon_filter(name, p):
    """Muon targets: 2-D weights other than embeddings and the output head (those, and every 1-D
    parameter, get AdamW)."""
    lname = name.lower()
    return p.dim() == 2 and not any(k in lname for k in ("embed", "lm_head", "output"))


class Muon(torch.optim.Optimizer):
    """Muon(model, lr=0.02, ns_backend="gram", ...): one C call for all Muon matrices and one for the rest.

    model_or_params: an nn.Module (parameters classified by `muon_filter(name, param)`; by default
    `default_muon_filter`, and nn.Embedding tables always go to AdamW) or an iterable of parameters /
    (name, parameter) pairs. Group 0 holds the Muon
    parameters (options lr, momentum), group 1 the AdamW ones (adamw_lr, adamw_betas, adamw_eps,
    adamw_weight_decay); LR schedulers act on these options as usual. Gradients must be contiguous and of
    one dtype per group (fp32, or bf16 for the Muon group). A step enqueues on the current CUDA stream.
    """

    def __init__(self, model_or_params, lr=0.02, momentum=0.95, ns_backend="gram", coefficients=POLAR_EXPRESS,
                 restart_iterations=DEFAULT_RESTARTS, eps=1e-7, adamw_lr=3e-4, adamw_betas=(0.9, 0.95),
                 adamw_eps=1e-8, adamw_weight_decay=0.0, muon_filter=None):
        if ns_backend not in BACKENDS:
            raise ValueError(f"ns_backend must be one of {sorted(BACKENDS)}")
        embedding_params = set()
        if isinstance(model_or_params, torch.nn.Module):
            named = list(model_or_params.named_parameters())
            # Embedding tables are AdamW parameters whatever they are called.
            for mod in model_or_params.modules():
                if isinstance(mod, torch.nn.Embedding):
                    embedding_params.update(id(q) for q in mod.parameters(recurse=False))
        else:
            named = [(item if isinstance(item, tuple) else (f"param{i}", item))
                     for i, item in enumerate(model_or_params)]
        if muon_filter is None:
            def flt(name, p):
                return id(p) not in embedding_params and default_muon_filter(name, p)
        else:
            flt = muon_filter
        muon, rest = [], []
        for name, p in named:
            if not p.requires_grad:
                continue
            if not (p.is_cuda and p.dtype == torch.float32 and p.is_contiguous()):
                raise ValueError(f"parameter {name}: Muon needs contiguous fp32 CUDA parameters")
            (muon if flt(name, p) else rest).append(p)
        for p in muon:
            if p.dim() != 2:
                raise ValueError("the Muon filter selected a parameter that is not 2-D")
        if not muon and not rest:
            raise ValueError("no trainable parameters")
        defaults = dict(lr=lr, momentum=momentum, adamw_lr=adamw_lr, adamw_betas=tuple(adamw_betas),
                        adamw_eps=adamw_eps, adamw_weight_decay=adamw_weight_decay)
        groups = []
        if muon:
            groups.append(dict(params=muon, use_muon=True))
        if rest:
            groups.append(dict(params=rest, use_muon=False))
        super().__init__(groups, defaults)
        self._ns = (tuple(tuple(float(v) for v in c) for c in coefficients), tuple(int(r) for r in restart_iterations),
                    ns_backend, float(eps))
        self._calls = {}  # group index -> (pointer key, prepared C call)

    def _prepared(self, gi, ps, build):
        key = tuple((p.data_ptr(), p.grad.data_ptr(), p.grad.dtype) for p in ps)
        cached = self._calls.get(gi)
        if cached is None or cached[0] != key:
            cached = (key, build())
            self._calls[gi] = cached
        return cached[1]

    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        coeffs, restarts, backend, eps = self._ns
        for gi, group in enumerate(self.param_groups):
            ps = [p for p in group["params"] if p.grad is not None]
            if not ps:
                continue
            if group["use_muon"]:
                moms = []
                for p in ps:
                    st = self.state[p]
                    if "momentum_buffer" not in st:
                        st["momentum_buffer"] = torch.zeros_like(p, dtype=torch.float32)
                    moms.append(st["momentum_buffer"])
                call = self._prepared(gi, ps, lambda: MuonStep(ps, [p.grad for p in ps], moms, coeffs, restarts,
                                                               backend, eps))
                call(lr=group["lr"], beta=group["momentum"])
            else:
                for p in ps:
                    st = self.state[p]
                    if "exp_avg" not in st:
                        st["exp_avg"] = torch.zeros_like(p, dtype=torch.float32)
                        st["exp_avg_sq"] = torch.zeros_like(p, dtype=torch.float32)
                group["step"] = group.get("step", 0) + 1
                call = self._prepared(gi, ps, lambda: AdamWStep(ps, [p.grad for p in ps],
                                                                [self.state[p]["exp_avg"] for p in ps],
                                                                [self.state[p]["exp_avg_sq"] for p in ps]))
                call(step=group["step"], lr=group["adamw_lr"], betas=group["adamw_betas"], eps=group["adamw_eps"],
                     weight_decay=group["adamw_weight_decay"])
        return loss
