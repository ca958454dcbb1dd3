"""GPU: dmuon_adamw_step against the float64 AdamW oracle over three steps.

Tolerance: the kernel works in fp32; m and v carry a few fp32 roundings (relative ~1e-7 each), and
the parameter change is compared as (p_t - p_0), whose error is dominated by storing p in fp32
(|p| / |step| x 2^-24, about 1e-6 here). 1e-5 relative Frobenius on p_t - p_0, m and v."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import adamw  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = 1e-5
HP = dict(lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01)


@pytest.fixture(scope="module")
def dm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_momentum_gb300 as dm
    return dm


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.mark.parametrize("gdtype", ["f32", "bf16"])
def test_adamw_matches_oracle(dm, gdtype):
    numels = [1, 7, 1000, 65536 + 3, 100000, 4096]
    P0 = [workloads.gaussian((n,), 0.02, 20 + i) for i, n in enumerate(numels)]
    Ps = [torch.from_numpy(p.copy()).cuda() for p in P0]
    Ms = [torch.zeros(n, dtype=torch.float32, device="cuda") for n in numels]
    Vs = [torch.zeros(n, dtype=torch.float32, device="cuda") for n in numels]
    Gd = [torch.empty(n, dtype=torch.bfloat16 if gdtype == "bf16" else torch.float32, device="cuda") for n in numels]
    step = dm.AdamWStep(Ps, Gd, Ms, Vs)
    ref = [(p.astype(np.float64), np.zeros(n), np.zeros(n)) for p, n in zip(P0, numels)]
    for t in range(1, 4):
        for i, n in enumerate(numels):
            g = workloads.gaussian((n,), 1e-3, 100 * t + i)
            if gdtype == "bf16":
                g, bits = workloads.round_to_bf16(g)
                Gd[i].copy_(torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16))
            else:
                Gd[i].copy_(torch.from_numpy(g).cuda())
            p, m, v = ref[i]
            ref[i] = adamw.adamw_step(p, g, m, v, HP["lr"], HP["betas"][0], HP["betas"][1], HP["eps"],
                                      HP["weight_decay"], t)
        step(t, **HP)
    dm.check_status()
    for i in range(len(numels)):
        p, m, v = ref[i]
        assert rel(Ps[i].cpu().numpy() - P0[i], p - P0[i]) <= TOL
        assert rel(Ms[i].cpu().numpy(), m) <= TOL
        assert rel(Vs[i].cpu().numpy(), v) <= TOL


def test_adamw_rejects_bad_step(dm):
    p = torch.zeros(8, device="cuda")
    with pytest.raises(dm.DmuonError):
        dm.adamw_step([p], [p.clone()], [p.clone()], [p.clone()], step=0)
