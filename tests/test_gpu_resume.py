"""GPU: checkpoint and resume give bit-identical training state (DMuon FAQ page, question
"有逐比特一致的收敛保证吗？" -- is convergence bit-for-bit reproducible: resuming from a checkpoint must
continue exactly as the uninterrupted run).

Two runs of two Muon steps from the same weights: one uninterrupted; the other takes step 1, copies W and
M to host memory (the checkpoint), drops its device buffers and the library's cached plan and workspace,
restores W and M into fresh device buffers and takes step 2 there. W and M after step 2 must be equal bit
for bit. Run for a grouped tensor-core plan (matrices wider than 128) and for a fused small-matrix plan."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_momentum_gb300 as dm
    return dm


def _step(dm, W, G, M, backend):
    dm.muon_step(W, G, M, lr=0.02, beta=0.95, coeffs=dm.POLAR_EXPRESS, restarts=(2,), backend=backend)


@pytest.mark.parametrize("shapes,backend", [
    ([(256, 1024), (1024, 256), (300, 700), (96, 520)], "gram"),
    ([(256, 1024), (640, 640)], "direct"),
    ([(128, 512), (512, 128), (100, 300)], "gram"),
])
def test_resume_is_bitwise_identical(dm, shapes, backend):
    W0 = [workloads.gaussian(s, 0.02, 10 + i) for i, s in enumerate(shapes)]
    G1 = [workloads.round_to_bf16(workloads.gaussian(s, 1e-3, 20 + i))[1] for i, s in enumerate(shapes)]
    G2 = [workloads.round_to_bf16(workloads.gaussian(s, 1e-3, 30 + i))[1] for i, s in enumerate(shapes)]

    def grads(bits):
        return [torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16) for b in bits]

    def fresh():
        return [torch.from_numpy(w).cuda() for w in W0], [torch.zeros(s, device="cuda") for s in shapes]

    Wa, Ma = fresh()
    _step(dm, Wa, grads(G1), Ma, backend)
    _step(dm, Wa, grads(G2), Ma, backend)
    dm.check_status()
    want = [t.cpu() for t in Wa + Ma]

    Wb, Mb = fresh()
    _step(dm, Wb, grads(G1), Mb, backend)
    dm.check_status()
    ckpt_w = [w.cpu() for w in Wb]
    ckpt_m = [m.cpu() for m in Mb]
    del Wb, Mb
    dm.release_workspace()
    torch.cuda.empty_cache()
    Wc = [w.cuda() for w in ckpt_w]
    Mc = [m.cuda() for m in ckpt_m]
    _step(dm, Wc, grads(G2), Mc, backend)
    dm.check_status()
    got = [t.cpu() for t in Wc + Mc]
    for i, (a, b) in enumerate(zip(want, got)):
        assert torch.equal(a, b), i
