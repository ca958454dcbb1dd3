"""GPU: failure detection without a fault. The library's kernels bound every mbarrier wait; a wait that
runs out records DMUON_ERR_TIMEOUT in the device status word and the kernel returns. The self-test makes
one such wait run out (a phase that nothing completes, 50 ms limit) and checks that the status is
reported once, that it clears, and that the context still computes correctly afterwards."""

import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_momentum_gb300 as dm
    return dm


def test_bounded_wait_times_out_and_reports(dm):
    dm.check_status()  # start clean
    t0 = time.perf_counter()
    dm.selftest_bounded_wait(0.05)
    with pytest.raises(dm.DmuonError) as ei:
        dm.check_status()
    elapsed = time.perf_counter() - t0
    assert ei.value.status == dm.ERR_TIMEOUT
    assert 0.04 <= elapsed < 2.0  # the wait ran to its limit and no further
    dm.check_status()  # the status word was cleared

    # the context is still usable: a GEMM after the timeout is correct
    rng = np.random.default_rng(3)
    a = rng.standard_normal((256, 320)).astype(np.float16)
    ad = torch.from_numpy(a).cuda()
    d = torch.empty((256, 256), dtype=torch.float16, device="cuda")
    dm.gemm_f16(ad, ad, d, b_trans=True)
    dm.check_status()
    want = a.astype(np.float64) @ a.astype(np.float64).T
    got = d.float().cpu().numpy()
    assert np.linalg.norm(got - want) <= 2e-3 * np.linalg.norm(want)


def test_workspace_limit_reports_oom_before_any_launch(dm):
    """A call whose plan needs more workspace than the set limit fails with DMUON_ERR_OOM and a message
    naming the limit, before anything is launched: no kernel ran (the per-launch record stays empty), and
    W and M are untouched. The same call goes through once the limit is lifted."""
    import workloads

    shapes = [(300, 1000), (1000, 300), (256, 1024)]
    W0 = [workloads.gaussian(s, 0.02, 40 + i) for i, s in enumerate(shapes)]
    M0 = [workloads.gaussian(s, 1e-3, 50 + i) for i, s in enumerate(shapes)]
    G = [torch.from_numpy(workloads.gaussian(s, 1e-3, 60 + i)).cuda() for i, s in enumerate(shapes)]
    W = [torch.from_numpy(w).cuda() for w in W0]
    M = [torch.from_numpy(m).cuda() for m in M0]
    need = dm.workspace_size(shapes, "gram")
    dm.release_workspace()  # the call below must plan and bind anew
    dm.set_workspace_limit(need // 2)
    dm.timing_enable(True)
    try:
        with pytest.raises(dm.DmuonError) as ei:
            dm.muon_step(W, G, M, lr=0.02, beta=0.95, coeffs=dm.YOU, restarts=(2,), backend="gram")
        assert ei.value.status == dm.ERR_OOM
        assert "exceeds the limit" in str(ei.value)
        assert dm.timing_read_launches() == []
    finally:
        dm.timing_enable(False)
        dm.set_workspace_limit(0)
    torch.cuda.synchronize()
    for w, w0, m, m0 in zip(W, W0, M, M0):
        assert np.array_equal(w.cpu().numpy(), w0)
        assert np.array_equal(m.cpu().numpy(), m0)
    dm.muon_step(W, G, M, lr=0.02, beta=0.95, coeffs=dm.YOU, restarts=(2,), backend="gram")
    dm.check_status()
    assert not np.array_equal(W[0].cpu().numpy(), W0[0])
