"""The pages' Python surface (newton_schulz, NewtonSchulz, Muon): CPU checks of the parameter split and
argument validation; GPU checks that each is exactly the C calls it wraps."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import newton_schulz_momentum_gb300 as dm  # noqa: E402
from newton_schulz_momentum_gb300 import optim  # noqa: E402


def _model():
    return torch.nn.Sequential(torch.nn.Embedding(100, 64), torch.nn.Linear(64, 192), torch.nn.LayerNorm(192),
                               torch.nn.Linear(192, 100, bias=False))


def test_default_filter_by_name():
    w = torch.zeros(4, 8)
    assert dm.default_muon_filter("layers.0.attn.q_proj.weight", w)
    assert not dm.default_muon_filter("model.embed_tokens.weight", w)
    assert not dm.default_muon_filter("lm_head.weight", w)
    assert not dm.default_muon_filter("layers.0.norm.weight", torch.zeros(8))


def test_cpu_parameters_rejected():
    with pytest.raises(ValueError):
        dm.Muon(_model())
    with pytest.raises(ValueError):
        dm.Muon([torch.zeros(4, 4)], ns_backend="bogus")


def test_newton_schulz_form_validated():
    with pytest.raises(ValueError):
        dm.NewtonSchulz("bogus")
    ns = dm.NewtonSchulz("direct", dm.YOU, [1, 3])
    assert ns.restart_iterations == (1, 3) and ns.backend == "direct"


@pytest.mark.gpu
def test_muon_optimizer_is_the_c_calls():
    """Two steps of Muon on a small model equal muon_step over the 2-D Linear weights plus adamw_step over
    the rest (embedding, biases, norm), bit for bit; an LR scheduler's change reaches the call."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.manual_seed(0)
    model = _model().cuda()
    ref = _model().cuda()
    ref.load_state_dict(model.state_dict())
    opt = dm.Muon(model, lr=0.02, momentum=0.95, ns_backend="gram", coefficients=dm.YOU, adamw_lr=1e-3)
    sched = torch.optim.lr_scheduler.StepLR(opt, step_size=1, gamma=0.5)
    assert len(opt.param_groups) == 2 and len(opt.param_groups[0]["params"]) == 2  # the two Linear weights
    named = dict(ref.named_parameters())
    muon_names = ["1.weight", "3.weight"]
    adam_names = ["0.weight", "1.bias", "2.weight", "2.bias"]
    moms = [torch.zeros_like(named[n]) for n in muon_names]
    ea = [torch.zeros_like(named[n]) for n in adam_names]
    eas = [torch.zeros_like(named[n]) for n in adam_names]
    lr = 0.02
    for step in (1, 2):
        gen = torch.Generator(device="cuda")
        gen.manual_seed(step)
        for (n, p), (_, q) in zip(model.named_parameters(), ref.named_parameters()):
            g = torch.randn(p.shape, generator=gen, device="cuda")
            p.grad = g.clone()
            q.grad = g.clone()
        opt.step()
        sched.step()
        dm.muon_step([named[n] for n in muon_names], [named[n].grad for n in muon_names], moms, lr=lr, beta=0.95,
                     coeffs=dm.YOU, restarts=(2,), backend="gram")
        dm.adamw_step([named[n] for n in adam_names], [named[n].grad for n in adam_names], ea, eas, step,
                      lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.0)
        lr *= 0.5
        dm.check_status()
        for (n, p), (_, q) in zip(model.named_parameters(), ref.named_parameters()):
            assert torch.equal(p, q), (step, n)


@pytest.mark.gpu
def test_newton_schulz_function_matches_ns():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import workloads
    g = torch.from_numpy(workloads.gaussian((300, 700), 1.0, 5)).cuda()
    keep = g.clone()
    out = dm.newton_schulz(g, coefficients=dm.YOU, restart_iterations=[2])
    assert torch.equal(g, keep)  # the input is not modified
    x = keep.clone()
    dm.ns(x, dm.YOU, (2,), "gram")
    assert torch.equal(out, x)
    assert torch.equal(dm.NewtonSchulz("gram", dm.YOU, (2,))(keep), x)
    dm.check_status()
    assert np.isfinite(out.cpu().numpy()).all()
