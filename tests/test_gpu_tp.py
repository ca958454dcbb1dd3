"""GPU: dmuon_ns_tp (the Gram form as tensor-parallel ranks compute it, emulated on one GPU) against the
oracle's split restatement at 2e-2 (the fp16 iteration bound), against the unsplit dmuon_ns, and run to
run bitwise."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import ns64  # noqa: E402

pytestmark = pytest.mark.gpu

TOL_NS = 2e-2


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
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def run(dm, g, fn, *args):
    x = torch.from_numpy(np.ascontiguousarray(g, dtype=np.float32)).cuda()
    fn(x, *args)
    dm.check_status()
    return x.cpu().numpy()


@pytest.mark.parametrize("shards", [1, 2, 3, 8])
@pytest.mark.parametrize("shape", [(256, 1024), (1024, 300), (300, 2000), (200, 200)])
def test_tp_matches_oracle_and_unsplit(dm, shards, shape):
    g = workloads.gaussian(shape, 1.0, 50 + shards)
    bounds = dm.shard_bounds(max(shape), shards)
    got = run(dm, g, lambda x: dm.ns_tp(x, shards, dm.YOU, (2,)))
    want = ns64.newton_schulz_tp(g, ns64.YOU, (2,), bounds, 1e-7)
    assert rel(got, want) <= TOL_NS
    unsplit = run(dm, g, lambda x: dm.ns(x, dm.YOU, (2,), "gram"))
    assert rel(got, unsplit) <= 5e-3  # the two differ only in fp32 summation order before fp16 rounding
    again = run(dm, g, lambda x: dm.ns_tp(x, shards, dm.YOU, (2,)))
    assert np.array_equal(got, again)


def test_tp_restart_lists(dm):
    g = workloads.gaussian((192, 1536), 1.0, 60)
    for rs in ((), (1, 3), (1, 2, 3, 4)):
        got = run(dm, g, lambda x: dm.ns_tp(x, 4, dm.YOU, rs))
        want = ns64.newton_schulz_tp(g, ns64.YOU, rs, dm.shard_bounds(1536, 4), 1e-7)
        assert rel(got, want) <= TOL_NS


@pytest.mark.slow
def test_tp_closed_form_top_tenth(dm):
    """The 2048 x 8192 top-10% closed-form matrix, POLAR_EXPRESS, split over 8 shards."""
    sigma = workloads.top_fraction_spectrum(2048, 0.1, 1.0, 1e-4)
    x, _, _ = workloads.closed_form_matrix(2048, 8192, sigma, 3)
    g = x.astype(np.float32)
    got = run(dm, g, lambda t: dm.ns_tp(t, 8, dm.POLAR_EXPRESS, (2,)))
    want = ns64.newton_schulz_tp(g, ns64.POLAR_EXPRESS, (2,), dm.shard_bounds(8192, 8), 1e-7)
    assert rel(got, want) <= TOL_NS


def test_tp_rejects_bad_shards(dm):
    x = torch.zeros((64, 256), device="cuda")
    with pytest.raises(dm.DmuonError):
        dm.ns_tp(x, 0)
    with pytest.raises(dm.DmuonError):
        dm.ns_tp(x, 17)  # 256 < 16 * 17
