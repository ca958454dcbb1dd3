"""GPU: the tcgen05 GEMM / SYRK building block (dmuon_gemm_f16) against float64 products of the same
fp16 operands. Shapes span several tiles, ragged edges, both B layouts, the symmetric (upper tiles
+ mirror) form, both tile widths (N <= 128 and N > 128) and the degenerate 1 x 1 case.

Tolerance: the kernel accumulates in fp32 and rounds the result to fp16 once, so the relative
Frobenius error is dominated by the final rounding (unit roundoff 2^-11, about 2.8e-4 RMS); 2e-3 leaves
room for fp32 accumulation over K up to 4096."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def dm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_momentum_gb300 as dm
    return dm


def _half(rng, rows, cols, scale, ld=None):
    ld = ld or ((cols + 7) // 8 * 8)
    a = (rng.standard_normal((rows, cols)) * scale).astype(np.float16)
    buf = torch.zeros((rows, ld), dtype=torch.float16, device="cuda")
    buf[:, :cols] = torch.from_numpy(a).cuda()
    return a, buf[:, :cols]


def _out(rows, cols):
    ld = (cols + 7) // 8 * 8
    return torch.full((rows, ld), float("nan"), dtype=torch.float16, device="cuda")[:, :cols]


def _rel(got, want):
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


@pytest.mark.parametrize("m,k", [(300, 520), (128, 64), (1, 7), (256, 1024), (1000, 100), (129, 4096)])
@pytest.mark.parametrize("sym", [True, False])
def test_xxt(dm, m, k, sym):
    rng = np.random.default_rng(m * 7 + k)
    x, xd = _half(rng, m, k, 1.0 / np.sqrt(k))
    d = _out(m, m)
    dm.gemm_f16(xd, xd, d, b_trans=True, symmetric=sym)
    dm.check_status()
    want = x.astype(np.float64) @ x.astype(np.float64).T
    got = d.float().cpu().numpy()
    assert np.isfinite(got).all(), "unwritten output elements"
    assert _rel(got, want) < TOL
    if sym:
        assert np.array_equal(got, got.T)


@pytest.mark.parametrize("m,n,k", [(200, 700, 200), (128, 512, 128), (300, 1000, 300), (64, 130, 64),
                                   (1024, 4096, 1024), (5, 9, 5)])
def test_b_row_major(dm, m, n, k):
    """D = A B with B stored K x N (the Q X and B X products): MN-major B tiles."""
    rng = np.random.default_rng(m + n + k)
    a, ad = _half(rng, m, k, 1.0 / np.sqrt(k))
    b, bd = _half(rng, k, n, 1.0)
    d = _out(m, n)
    dm.gemm_f16(ad, bd, d, b_trans=False)
    dm.check_status()
    want = a.astype(np.float64) @ b.astype(np.float64)
    got = d.float().cpu().numpy()
    assert np.isfinite(got).all()
    assert _rel(got, want) < TOL


@pytest.mark.parametrize("b_trans", [True, False])
def test_epilogue_scalars(dm, b_trans):
    """v = alpha * acc + beta * E + gamma * I (the recipes Z = b R + c R^2 and Q = Z + a I use these)."""
    rng = np.random.default_rng(5)
    m, k = 260, 260
    a, ad = _half(rng, m, k, 1.0 / np.sqrt(k))
    b, bd = _half(rng, m, k, 1.0)
    e, ed = _half(rng, m, m, 1.0)
    d = _out(m, m)
    dm.gemm_f16(ad, bd, d, b_trans=b_trans, e=ed, alpha=-0.75, beta=2.5, gamma=3.25)
    dm.check_status()
    bop = b.astype(np.float64).T if b_trans else b.astype(np.float64)
    want = -0.75 * (a.astype(np.float64) @ bop) + 2.5 * e.astype(np.float64) + 3.25 * np.eye(m)
    assert _rel(d.float().cpu().numpy(), want) < TOL


def test_symmetric_square_of_symmetric(dm):
    """R^2 for a symmetric R (the SYRK form used for R^2 and A^2), with the Z epilogue."""
    rng = np.random.default_rng(6)
    m = 384
    g = rng.standard_normal((m, 2 * m)) / np.sqrt(2 * m)
    r = (g @ g.T).astype(np.float16)
    rd = torch.from_numpy(r).cuda()
    d = _out(m, m)
    dm.gemm_f16(rd, rd, d, b_trans=True, e=rd, alpha=1.2, beta=-3.0, symmetric=True)
    dm.check_status()
    r64 = r.astype(np.float64)
    want = 1.2 * (r64 @ r64) - 3.0 * r64
    got = d.float().cpu().numpy()
    assert _rel(got, want) < TOL and np.array_equal(got, got.T)


def test_deterministic(dm):
    rng = np.random.default_rng(7)
    x, xd = _half(rng, 700, 1500, 0.03)
    d1, d2 = _out(700, 700), _out(700, 700)
    dm.gemm_f16(xd, xd, d1, symmetric=True)
    dm.gemm_f16(xd, xd, d2, symmetric=True)
    dm.check_status()
    assert torch.equal(d1, d2)


@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("m,k", [(300, 520), (512, 256)])
def test_overflow_reported(dm, m, k, sym):
    """A result past the fp16 range raises the NONFINITE status: here only row and column m-1 of X Xᵀ
    (the ragged last tile when m = 300; in the mirrored part when symmetric) exceed 65504."""
    rng = np.random.default_rng(m + k)
    x, xd = _half(rng, m, k, 1.0 / np.sqrt(k))
    xd[m - 1, :] = 64.0  # D[m-1][m-1] = 4096 k > 65504
    d = _out(m, m)
    dm.gemm_f16(xd, xd, d, b_trans=True, symmetric=sym)
    with pytest.raises(dm.DmuonError) as ei:
        dm.check_status()
    assert ei.value.status == dm.ERR_NONFINITE
    dm.check_status()  # the word was cleared


@pytest.mark.parametrize("b_trans", [True, False])
def test_nan_reported(dm, b_trans):
    """A NaN operand element propagates into its output row and is reported."""
    rng = np.random.default_rng(21)
    m, n, k = 260, 300, 264
    a, ad = _half(rng, m, k, 1.0 / np.sqrt(k))
    b, bd = _half(rng, n, k, 1.0) if b_trans else _half(rng, k, n, 1.0)
    ad[137, 5] = float("nan")
    d = _out(m, n)
    dm.gemm_f16(ad, bd, d, b_trans=b_trans)
    with pytest.raises(dm.DmuonError) as ei:
        dm.check_status()
    assert ei.value.status == dm.ERR_NONFINITE
    dm.check_status()


def test_large_finite_not_reported(dm):
    """Results just inside the fp16 range (up to 65504 after rounding) are not flagged."""
    m, k = 256, 64
    xd = torch.full((m, k), 32.0, dtype=torch.float16, device="cuda")  # every element of X Xᵀ: 65536 k / 64
    xd[:, 63] = 0.0
    xd[:, 62] = 31.0  # row sums of squares: 62 * 1024 + 961 = 64449
    d = _out(m, m)
    dm.gemm_f16(xd, xd, d, b_trans=True, symmetric=True)
    dm.check_status()
    got = d.float().cpu().numpy()
    assert np.all(got == 64448.0)  # 64449 rounds to the fp16 neighbour 64448
