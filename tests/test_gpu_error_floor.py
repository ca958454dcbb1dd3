"""The GPU's Newton-Schulz error against the float64 oracle, held to the error an fp16 iteration must make.

oracle/fp16_model.py plays the same iteration with fp16-stored intermediates and fp32 accumulation: its
distance from the oracle is the floor that fp16 storage sets ("Newton-Schulz 变体", section "精度流水线":
fp32 normalisation, fp16 iteration). The kernels' error, measured against the same oracle on the same input,
must lie between 0.5 and 1.5 times that floor. Above it lie a kernel that accumulates in fp16, rounds a step's
scalar recipe before applying it, or loses a restart, and also subtler slips: reading the second operand of
R^2, Z R and S Z transposed (the same products in exact arithmetic, not for fp16-stored values) gives about
2.2 times the floor on a 256 x 1024 Gram iteration (tests/test_fp16_model.py). Far below it, the kernel would
not be running the fp16 pipeline at all. The per-matrix floors are noisy where a coefficient table amplifies
rounding (POLAR_EXPRESS on Gaussians), hence the wider lower bound. The fixed 2e-2 / 6e-2 tolerances of the
parity tests sit above these floors; this file says how far above.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import fp16_model, ns64  # noqa: E402

pytestmark = pytest.mark.gpu

EPS = 1e-7
LOW, HIGH = 0.5, 1.5


@pytest.fixture(scope="module")
def dm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_momentum_gb300 as dm
    return dm


def rel(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def tables(dm, name):
    return getattr(dm, name), getattr(ns64, name)


def assert_at_floor(gpu_err, g, coeffs, restarts, backend, where):
    want = ns64.newton_schulz(g, coeffs, restarts, backend, EPS)
    floor = rel(fp16_model.newton_schulz(g.astype(np.float32), coeffs, restarts, backend, EPS), want)
    ratio = gpu_err(want) / floor
    print(f"{where}: floor {floor:.3e}, kernel / floor {ratio:.3f}")
    assert LOW <= ratio <= HIGH, (where, floor, ratio)


@pytest.mark.parametrize("backend", ["direct", "gram"])
@pytest.mark.parametrize("shape,table", [((256, 1024), "YOU"), ((200, 600), "YOU"), ((129, 700), "YOU"),
                                         ((1024, 4096), "YOU"), ((4096, 1024), "POLAR_EXPRESS"),
                                         ((300, 1000), "POLAR_EXPRESS")])
def test_dmuon_ns_at_the_fp16_floor(dm, shape, table, backend):
    """One matrix through dmuon_ns: the 256 x 1024 parity case and two ragged matrices with m <= 256 (symmetric
    products computed in full), a 1024 x 4096 and a tall 4096 x 1024 (symmetric products computed once and
    mirrored), and a ragged 300 x 1000."""
    g = workloads.gaussian(shape, 1.0, 7 + shape[0])
    tab_dm, tab = tables(dm, table)
    x = torch.from_numpy(g.astype(np.float32)).cuda()
    dm.ns(x, tab_dm, (2,), backend, EPS)
    dm.check_status()
    got = x.cpu().numpy()
    assert_at_floor(lambda want: rel(got, want), g, tab, (2,), backend, f"{shape} {table} {backend}")


@pytest.mark.parametrize("table", ["YOU", "POLAR_EXPRESS"])
def test_small_fused_kernel_at_the_fp16_floor(dm, table):
    """Matrices of the 2560-matrix small set (128 x 512 and 512 x 128 gradients, N(0, 1e-3^2), momentum from
    zero, Gram with restart [2]) through one Muon step in the fused small-matrix kernel. With POLAR_EXPRESS the
    floor is about 5e-2 on these matrices: that is the fp16 pipeline's own error, not the kernel's."""
    shapes = workloads.small_set_shapes()
    pick = [0, 97, 1500, 2047, 2048, 2300, 2559]
    G = [workloads.gaussian(shapes[i], 1e-3, 1000 + i) for i in pick]
    W = [workloads.gaussian(shapes[i], 0.02, 5000 + i) for i in pick]
    Wd = [torch.from_numpy(w).cuda() for w in W]
    Gd = [torch.from_numpy(g).cuda() for g in G]
    Md = [torch.zeros(shapes[i], dtype=torch.float32, device="cuda") for i in pick]
    tab_dm, tab = tables(dm, table)
    dm.muon_step(Wd, Gd, Md, lr=0.02, beta=0.95, coeffs=tab_dm, restarts=(2,), backend="gram")
    dm.check_status()
    for k, i in enumerate(pick):
        upd = (W[k].astype(np.float64) - Wd[k].cpu().numpy().astype(np.float64)) / 0.02
        # momentum from zero: M = G exactly, the input of both the oracle and the model
        assert_at_floor(lambda want: rel(upd, want), G[k], tab, (2,), "gram", f"small[{i}] {shapes[i]} {table}")


@pytest.mark.slow
def test_top_tenth_closed_form_at_the_fp16_floor(dm):
    """2048 x 8192 with 205 singular values at 1 and the rest at 1e-4, POLAR_EXPRESS, Gram with restart [2]."""
    sigma = workloads.top_fraction_spectrum(2048, 0.1, 1.0, 1e-4)
    x, _, _ = workloads.closed_form_matrix(2048, 8192, sigma, 3)
    g = x.astype(np.float32)
    xd = torch.from_numpy(g).cuda()
    dm.ns(xd, dm.POLAR_EXPRESS, (2,), "gram", EPS)
    dm.check_status()
    got = xd.cpu().numpy()
    assert_at_floor(lambda want: rel(got, want), g.astype(np.float64), ns64.POLAR_EXPRESS, (2,), "gram",
                    "2048x8192 top tenth")


@pytest.mark.slow
@pytest.mark.parametrize("backend", ["gram", "direct"])
def test_llama_shapes_at_the_fp16_floor(dm, backend):
    """One Muon step over the four Llama-3-8B projection shapes (q/o 4096 x 4096, k/v 1024 x 4096, gate/up
    14336 x 4096, down 4096 x 14336), bf16 gradients N(0, 1e-3^2), momentum from zero, POLAR_EXPRESS: the
    grouped launches with 256 x 256 CTA-pair tiles and mirrored symmetric products that the 8B step runs."""
    shapes = [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)]
    G = [workloads.round_to_bf16(workloads.gaussian(s, 1e-3, 700 + i))[0] for i, s in enumerate(shapes)]
    W = [workloads.gaussian(s, 0.02, 800 + i) for i, s in enumerate(shapes)]
    Wd = [torch.from_numpy(w).cuda() for w in W]
    Gd = [torch.from_numpy(g).cuda().to(torch.bfloat16) for g in G]
    Md = [torch.zeros(s, dtype=torch.float32, device="cuda") for s in shapes]
    dm.muon_step(Wd, Gd, Md, lr=0.02, beta=0.95, coeffs=dm.POLAR_EXPRESS, restarts=(2,), backend=backend)
    dm.check_status()
    for k, s in enumerate(shapes):
        upd = (W[k].astype(np.float64) - Wd[k].cpu().numpy().astype(np.float64)) / 0.02
        # momentum from zero: M = G (the bf16 values, exact in fp32)
        assert_at_floor(lambda want: rel(upd, want), G[k], ns64.POLAR_EXPRESS, (2,), backend, f"{s} {backend}")
