"""Graph replay of repeated calls: bit-identical to direct launches, reading fresh data every call, and
falling back to direct launches when an argument changes, after a workspace release or under timing."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import ns64  # noqa: E402

pytestmark = pytest.mark.gpu

EPS = 1e-7


@pytest.fixture(scope="module")
def dm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_momentum_gb300 as dm
    yield dm
    dm.set_graph_replay(True)


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_steps(dm, shapes, replay, calls=4, lr=None):
    """`calls` Muon steps (YOU coefficients, Gram, restart [2]) over the same buffers, with new gradient
    values copied in before every call. Returns W and M after each call (host copies)."""
    lr = lr or (0.02,) * calls
    dm.set_graph_replay(replay)
    dm.release_workspace()
    W = [cuda(workloads.gaussian(s, 0.02, 10 + i)) for i, s in enumerate(shapes)]
    M = [torch.zeros(s, dtype=torch.float32, device="cuda") for s in shapes]
    G = [torch.empty(s, dtype=torch.float32, device="cuda") for s in shapes]
    out = []
    for c in range(calls):
        for i, s in enumerate(shapes):
            G[i].copy_(cuda(workloads.gaussian(s, 1e-3, 100 * c + i)))
        dm.muon_step(W, G, M, lr=lr[c], beta=0.95, coeffs=dm.YOU, restarts=(2,), backend="gram")
        dm.check_status()
        out.append(([w.cpu().numpy() for w in W], [m.cpu().numpy() for m in M]))
    return out


@pytest.mark.parametrize("shapes", [[(256, 1024), (1024, 300), (200, 200)], [(128, 512), (512, 128)] * 4],
                         ids=["grouped-gemm", "fused-small"])
def test_replay_is_bit_identical_and_reads_fresh_data(dm, shapes):
    direct = run_steps(dm, shapes, replay=False)
    replay = run_steps(dm, shapes, replay=True)
    for c in range(len(direct)):
        for a, b in zip(direct[c][0] + direct[c][1], replay[c][0] + replay[c][1]):
            assert np.array_equal(a, b), c
    # and the replayed calls still follow the oracle (new gradients every call)
    w_prev = workloads.gaussian(shapes[0], 0.02, 10)
    m_prev = np.zeros(shapes[0])
    for c in range(len(replay)):
        g = workloads.gaussian(shapes[0], 1e-3, 100 * c)
        ref = ns64.muon_step(w_prev, g, m_prev, 0.02, 0.95, ns64.YOU, (2,), "gram", EPS)
        upd = (w_prev - replay[c][0][0].astype(np.float64)) / 0.02
        assert np.linalg.norm(upd - ref["O"]) / np.linalg.norm(ref["O"]) <= 2e-2, c
        w_prev, m_prev = replay[c][0][0].astype(np.float64), ref["M"]


def test_changed_learning_rate_is_honoured(dm):
    shapes = [(256, 1024), (300, 700)]
    lrs = (0.02, 0.02, 0.02, 0.005)  # captured on the second call, replayed on the third, then changed
    direct = run_steps(dm, shapes, replay=False, lr=lrs)
    replay = run_steps(dm, shapes, replay=True, lr=lrs)
    for a, b in zip(direct[-1][0] + direct[-1][1], replay[-1][0] + replay[-1][1]):
        assert np.array_equal(a, b)


def test_ns_replay_and_workspace_release(dm):
    dm.set_graph_replay(True)
    x = torch.empty(256, 1024, device="cuda")
    for c in range(4):
        if c == 2:
            dm.release_workspace()  # the captured graph goes with the workspace
        g = workloads.gaussian((256, 1024), 1.0, 40 + c)
        x.copy_(cuda(g))
        dm.ns(x, dm.YOU, (2,), "gram", EPS)
        dm.check_status()
        want = ns64.newton_schulz(g, ns64.YOU, (2,), "gram", EPS)
        got = x.cpu().numpy()
        assert np.linalg.norm(got - want) / np.linalg.norm(want) <= 2e-2, c


def test_timing_launches_directly(dm):
    """With per-launch timing on, every kernel is still recorded on repeated calls (no replay)."""
    dm.set_graph_replay(True)
    x = torch.randn(256, 1024, device="cuda")
    for _ in range(2):
        dm.ns(x, dm.YOU, (2,), "gram", EPS)
    dm.timing_enable(True)
    for _ in range(3):
        dm.ns(x, dm.YOU, (2,), "gram", EPS)
    torch.cuda.synchronize()
    launches = dm.timing_read_launches()
    dm.timing_enable(False)
    dm.check_status()
    assert len(launches) == 3 * 20


def test_caller_graph_capture_holds_the_kernels(dm):
    """A caller capturing the call into a CUDA graph of its own (after the library has captured one for
    itself) gets the launches in its graph; replaying it reads fresh gradients, bit-identical to direct."""
    shapes = [(256, 1024), (1024, 300)]
    direct = run_steps(dm, shapes, replay=False, calls=5)
    dm.set_graph_replay(True)
    dm.release_workspace()
    W = [cuda(workloads.gaussian(s, 0.02, 10 + i)) for i, s in enumerate(shapes)]
    M = [torch.zeros(s, dtype=torch.float32, device="cuda") for s in shapes]
    G = [torch.empty(s, dtype=torch.float32, device="cuda") for s in shapes]
    s = torch.cuda.Stream()

    def load(c):
        for i, sh in enumerate(shapes):
            G[i].copy_(cuda(workloads.gaussian(sh, 1e-3, 100 * c + i)))

    def call():
        dm.muon_step(W, G, M, lr=0.02, beta=0.95, coeffs=dm.YOU, restarts=(2,), backend="gram",
                     stream=s.cuda_stream)

    for c in range(3):  # direct, library capture, library replay
        load(c)
        with torch.cuda.stream(s):
            call()
        torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call()
    for c in range(3, 5):
        load(c)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        dm.check_status()
        for a, b in zip(direct[c][0] + direct[c][1], [w.cpu().numpy() for w in W] + [m.cpu().numpy() for m in M]):
            assert np.array_equal(a, b), c
