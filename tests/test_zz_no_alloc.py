"""GPU: the allocation-free entry point dmuon_momentum_normalize_noalloc, called through the C ABI.

Some callers cannot let a library call cudaMalloc: their device memory is owned by a framework's
caching allocator or a fixed memory plan, or they cannot afford the device-wide synchronisation an
allocation may cause. This entry point keeps its scratch in a fixed array inside the library's device
image instead. The test checks that two calls in a row (the second one finding the first one's data in
that shared scratch) give the same momentum, norm and fp16 X as the workspace-based
dmuon_momentum_normalize, within the tolerances of the other parity tests: 1e-5 relative for the fp32
momentum and norm, 1e-3 relative Frobenius for the fp16 X -- and the same against the CPU float64 oracle.
A call without a gradient (the norm and X of M alone) is checked the same way, and the size limit is
checked to be enforced before anything runs. This file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import ns64  # noqa: E402

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-5
TOL_X = 1e-3


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


def _noalloc(dm, g, gdtype, m, x, norm):
    stream = torch.cuda.current_stream().cuda_stream
    rc = dm.lib().dmuon_momentum_normalize_noalloc(
        None if g is None else ctypes.c_void_p(g.data_ptr()), gdtype, ctypes.c_void_p(m.data_ptr()), m.shape[0], m.shape[1],
        ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(norm.data_ptr()), 0.95, 1e-7, ctypes.c_void_p(stream))
    assert rc == dm.OK, dm.lib().dmuon_last_error().decode()


@pytest.mark.parametrize("shape,dtype", [((1000, 3000), "bf16"), ((4096, 1030), "f32"), ((7, 5), "f32")])
def test_noalloc_matches_workspace_path_twice(dm, shape, dtype):
    r, c = shape
    g1 = workloads.gaussian(shape, 1e-3, 301)
    g2 = workloads.gaussian(shape, 1e-3, 302)
    m0 = workloads.gaussian(shape, 1e-3, 303)
    if dtype == "bf16":
        grads = [torch.from_numpy(workloads.round_to_bf16(g)[1].view(np.int16)).cuda().view(torch.bfloat16)
                 for g in (g1, g2)]
        gdtype = dm.BF16
    else:
        grads = [torch.from_numpy(g).cuda() for g in (g1, g2)]
        gdtype = dm.F32
    m_ref = torch.from_numpy(m0).cuda()
    m_new = m_ref.clone()
    xs = (min(r, c), max(r, c))
    m_host = m0.astype(np.float64)
    for g, gh in zip(grads, (g1, g2)):  # two calls in a row on the same shared scratch
        x_ref = torch.empty(xs, dtype=torch.float16, device="cuda")
        x_new = torch.full(xs, float("nan"), dtype=torch.float16, device="cuda")
        n_ref = torch.empty(1, dtype=torch.float32, device="cuda")
        n_new = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
        dm.momentum_normalize([g], [m_ref], [x_ref], n_ref, beta=0.95, eps=1e-7)
        _noalloc(dm, g, gdtype, m_new, x_new, n_new)
        dm.check_status()
        assert rel(m_new.cpu().numpy(), m_ref.cpu().numpy()) <= TOL_F32
        assert abs(n_new.item() - n_ref.item()) <= TOL_F32 * n_ref.item()
        assert rel(x_new.float().cpu().numpy(), x_ref.float().cpu().numpy()) <= TOL_X
        # the CPU float64 oracle, fed the gradient values the GPU saw and the momentum before the call
        g_seen = workloads.round_to_bf16(gh)[0] if dtype == "bf16" else gh
        m_want = ns64.momentum(m_host, g_seen, 0.95)
        x_want, s_want = ns64.normalise(m_want, 1e-7)
        x_want, _ = ns64.orient(x_want)
        assert rel(m_new.cpu().numpy(), m_want) <= TOL_F32
        assert abs(n_new.item() - s_want) <= TOL_F32 * s_want
        assert rel(x_new.float().cpu().numpy(), x_want) <= TOL_X
        m_host = m_new.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("shape", [(333, 77), (64, 4096)])
def test_noalloc_without_gradient_twice(dm, shape):
    """grad = NULL: M is only read; its norm and X match the workspace path's norm-only call and the
    oracle, on two calls in a row."""
    r, c = shape
    xs = (min(r, c), max(r, c))
    for seed in (401, 402):
        m0 = workloads.gaussian(shape, 2.0, seed)
        m = torch.from_numpy(m0).cuda()
        x_ref = torch.empty(xs, dtype=torch.float16, device="cuda")
        n_ref = torch.empty(1, dtype=torch.float32, device="cuda")
        dm.momentum_normalize(None, [m], [x_ref], n_ref, beta=0.95, eps=1e-7)
        x_new = torch.full(xs, float("nan"), dtype=torch.float16, device="cuda")
        n_new = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
        _noalloc(dm, None, dm.F32, m, x_new, n_new)
        dm.check_status()
        assert np.array_equal(m.cpu().numpy(), m0)  # untouched
        assert abs(n_new.item() - n_ref.item()) <= TOL_F32 * n_ref.item()
        assert rel(x_new.float().cpu().numpy(), x_ref.float().cpu().numpy()) <= TOL_X
        x_want, s_want = ns64.normalise(m0.astype(np.float64), 1e-7)
        x_want, _ = ns64.orient(x_want)
        assert abs(n_new.item() - s_want) <= TOL_F32 * s_want
        assert rel(x_new.float().cpu().numpy(), x_want) <= TOL_X


def test_noalloc_rejects_oversized_matrix(dm):
    m = torch.zeros((1, 16), dtype=torch.float32, device="cuda")
    x = torch.zeros((1, 16), dtype=torch.float16, device="cuda")
    n = torch.zeros(1, dtype=torch.float32, device="cuda")
    rc = dm.lib().dmuon_momentum_normalize_noalloc(
        None, dm.F32, ctypes.c_void_p(m.data_ptr()), 16385, 16385, ctypes.c_void_p(x.data_ptr()),
        ctypes.c_void_p(n.data_ptr()), 0.95, 1e-7, None)
    assert rc == dm.ERR_INVALID_ARG
    assert "DMUON_NOALLOC_MAX_ELEMS" in dm.lib().dmuon_last_error().decode()
