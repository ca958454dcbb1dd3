"""GPU: dmuon_muon_step_host -- the step with its gradients copied in from host memory, the copies
pipelined against the computation in groups of matrices.

The call must give bit-identical W, M and norms to copying every gradient to the device and calling
dmuon_muon_step (grouping changes the launch schedule, never a matrix's arithmetic): for every group
count (one, several, more groups than matrices, the library's choice), over consecutive steps that
refill the same host buffers, when the group count changes between calls, from pinned and from
pageable host memory, with bf16 and fp32 gradients, and for the fused small-matrix plan. One case is
also checked against the float64 oracle directly; the device path itself is pinned to the oracle in
test_gpu_parity.py. The YOU coefficients are used throughout: the printed POLAR_EXPRESS polynomials
amplify normalised singular values above ~0.02, so thin Gaussian matrices such as 8 x 1000 overflow
fp16 under them (reported as NONFINITE, in the oracle too), which says nothing about the pipeline."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import ns64  # noqa: E402

pytestmark = pytest.mark.gpu

EPS = 1e-7
SHAPES = [(520, 264), (264, 1040), (1024, 256), (96, 520), (300, 300), (512, 2048), (130, 130), (2048, 512),
          (8, 1000), (640, 128)]
SMALL = [(128, 512), (512, 128), (100, 300), (64, 64), (7, 1)]


@pytest.fixture(scope="module")
def dm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_momentum_gb300 as dm
    return dm


def _grads(shapes, seed, dtype):
    return [torch.from_numpy(workloads.gaussian(s, 1.0, seed + i)).to(dtype) for i, s in enumerate(shapes)]


def _state(shapes, dtype):
    W = [torch.from_numpy(workloads.gaussian(s, 0.02, 500 + i)).cuda() for i, s in enumerate(shapes)]
    M = [torch.zeros(s, dtype=torch.float32, device="cuda") for s in shapes]
    G = [torch.empty(s, dtype=dtype, device="cuda") for s in shapes]
    norms = torch.empty(len(shapes), dtype=torch.float32, device="cuda")
    return W, M, G, norms


def _reference(dm, shapes, steps_grads, dtype, backend="gram"):
    """Copy every gradient to the device, then the device-buffer call."""
    W, M, G, norms = _state(shapes, dtype)
    out = []
    for grads in steps_grads:
        for gd, gh in zip(G, grads):
            gd.copy_(gh)
        dm.muon_step(W, G, M, lr=0.02, beta=0.95, coeffs=dm.YOU, restarts=(2,), backend=backend,
                     norms_out=norms)
        out.append(norms.cpu())
    dm.check_status()
    return [w.cpu() for w in W], [m.cpu() for m in M], out


def _pipelined(dm, shapes, steps_grads, dtype, groups, pinned=True, backend="gram"):
    """pinned: True, False, or "mixed" (every other host buffer page-locked)."""
    W, M, G, norms = _state(shapes, dtype)
    H = [torch.empty(s, dtype=dtype, pin_memory=(i % 2 == 0) if pinned == "mixed" else pinned)
         for i, s in enumerate(shapes)]
    out = []
    groups_seq = groups if isinstance(groups, (list, tuple)) else [groups] * len(steps_grads)
    for grads, g in zip(steps_grads, groups_seq):
        torch.cuda.synchronize()  # the previous call has read H before the host refills it
        for h, src in zip(H, grads):
            h.copy_(src)
        step = dm.MuonStep(W, G, M, coeffs=dm.YOU, restarts=(2,), backend=backend, norms_out=norms,
                           host_grads=H, groups=g)
        step(lr=0.02, beta=0.95)
        out.append(norms.cpu())
    dm.check_status()
    return [w.cpu() for w in W], [m.cpu() for m in M], out


def _equal(a, b):
    return all(torch.equal(x, y) for x, y in zip(a[0] + a[1] + a[2], b[0] + b[1] + b[2]))


@pytest.mark.parametrize("groups", [1, 2, 3, 5, 0, 64])
def test_pipelined_matches_device_call(dm, groups):
    steps = [_grads(SHAPES, 100, torch.bfloat16), _grads(SHAPES, 200, torch.bfloat16)]
    ref = _reference(dm, SHAPES, steps, torch.bfloat16)
    got = _pipelined(dm, SHAPES, steps, torch.bfloat16, groups)
    assert _equal(ref, got)


def test_group_count_changes_between_calls(dm):
    steps = [_grads(SHAPES, 300 + 100 * k, torch.bfloat16) for k in range(3)]
    ref = _reference(dm, SHAPES, steps, torch.bfloat16)
    got = _pipelined(dm, SHAPES, steps, torch.bfloat16, [2, 4, 1])
    assert _equal(ref, got)


def test_pageable_host_memory_fp32(dm):
    steps = [_grads(SHAPES, 700, torch.float32), _grads(SHAPES, 800, torch.float32)]
    ref = _reference(dm, SHAPES, steps, torch.float32)
    got = _pipelined(dm, SHAPES, steps, torch.float32, 3, pinned=False)
    assert _equal(ref, got)


@pytest.mark.parametrize("backend", ["auto", "direct"])
def test_other_backends_pipelined(dm, backend):
    steps = [_grads(SHAPES, 900, torch.bfloat16)]
    ref = _reference(dm, SHAPES, steps, torch.bfloat16, backend=backend)
    got = _pipelined(dm, SHAPES, steps, torch.bfloat16, 3, backend=backend)
    assert _equal(ref, got)


def test_small_fused_plan_with_host_gradients(dm):
    steps = [_grads(SMALL, 1000, torch.float32), _grads(SMALL, 1100, torch.float32)]
    ref = _reference(dm, SMALL, steps, torch.float32)
    got = _pipelined(dm, SMALL, steps, torch.float32, 3)
    assert _equal(ref, got)


def test_pipelined_against_oracle(dm):
    """One step from zero momentum straight against the float64 oracle (tolerances of test_gpu_parity)."""
    shapes = [(264, 1040), (1024, 256), (300, 300)]
    grads = _grads(shapes, 1200, torch.float32)
    W0 = [workloads.gaussian(s, 0.02, 500 + i) for i, s in enumerate(shapes)]
    W, M, norms_out = _pipelined(dm, shapes, [grads], torch.float32, 2)
    for i, s in enumerate(shapes):
        ref = ns64.muon_step(W0[i].astype(np.float64), grads[i].numpy(), np.zeros(s), 0.02, 0.95,
                             ns64.YOU, (2,), "gram", EPS)
        m = M[i].numpy().astype(np.float64)
        assert np.linalg.norm(m - ref["M"]) <= 1e-5 * np.linalg.norm(ref["M"])
        assert abs(float(norms_out[0][i]) - ref["norm"]) <= 1e-5 * ref["norm"]
        upd = (W0[i].astype(np.float64) - W[i].numpy().astype(np.float64)) / 0.02
        assert np.linalg.norm(upd - ref["O"]) <= 2e-2 * np.linalg.norm(ref["O"])


# Many small matrices take the one-launch gather out of host memory instead of a copy per matrix.
MANY_SMALL = [(96, 200), (200, 96), (64, 64), (128, 512), (7, 1), (33, 130)] * 12   # fused small-matrix plan
MANY_MEDIUM = [(300, 264), (264, 520), (256, 256)] * 24                           # grouped GEMM plan


@pytest.mark.parametrize("pinned", [True, False, "mixed"])
@pytest.mark.parametrize("shapes", [MANY_SMALL, MANY_MEDIUM], ids=["fused", "grouped"])
def test_many_small_matrices_gather(dm, shapes, pinned):
    steps = [_grads(shapes, 1300, torch.float32), _grads(shapes, 1400, torch.float32)]
    ref = _reference(dm, shapes, steps, torch.float32)
    got = _pipelined(dm, shapes, steps, torch.float32, 0, pinned=pinned)
    assert _equal(ref, got)
