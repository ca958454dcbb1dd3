"""GPU parity of the whole path against the CPU float64 oracle, through the C ABI.

Tolerances (stated per quantity, per matrix):
  * fp32 momentum M and its Frobenius norm: relative error <= 1e-5 (fp32 arithmetic against float64).
  * fp16 X = M / (||M|| + eps): relative Frobenius error <= 1e-3 (one fp16 rounding, 2^-11).
  * Newton-Schulz output O (and the update (W0 - W) / lr): relative Frobenius error <= 2e-2, the
    bound for the fp16 iteration path.
Inputs come from workloads/ (seeded NumPy), never from the CUDA path.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import ns64  # noqa: E402

pytestmark = pytest.mark.gpu

EPS = 1e-7
TOL_NS = 2e-2
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


def rel(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# ------------------------------------------------------------------------------- momentum / normalise


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_momentum_normalize(dm, dtype):
    shapes = [(256, 1024), (1024, 256), (300, 1000), (1000, 300), (7, 5), (1, 1), (65, 129), (4096, 1030)]
    grads_h, moms_h, grads_d, moms_d, xs = [], [], [], [], []
    for i, (r, c) in enumerate(shapes):
        g = workloads.gaussian((r, c), 1e-3, 40 + i)
        m0 = workloads.gaussian((r, c), 1e-3, 60 + i)
        if dtype == "bf16":
            g, bits = workloads.round_to_bf16(g)
            gd = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
        else:
            gd = cuda(g)
        grads_h.append(g)
        moms_h.append(m0)
        grads_d.append(gd)
        moms_d.append(cuda(m0))
        xs.append(torch.empty((min(r, c), max(r, c)), dtype=torch.float16, device="cuda"))
    norms = torch.empty(len(shapes), dtype=torch.float32, device="cuda")
    dm.momentum_normalize(grads_d, moms_d, xs, norms, beta=0.95, eps=EPS)
    dm.check_status()
    nh = norms.cpu().numpy()
    for i, (g, m0) in enumerate(zip(grads_h, moms_h)):
        m = ns64.momentum(m0, g, 0.95)
        x, s = ns64.normalise(m, EPS)
        x, _ = ns64.orient(x)
        assert rel(moms_d[i].cpu().numpy(), m) <= TOL_F32
        assert abs(nh[i] - s) <= TOL_F32 * s
        assert rel(xs[i].float().cpu().numpy(), x) <= TOL_X


def test_norm_only_when_no_gradient(dm):
    m0 = workloads.gaussian((333, 77), 2.0, 5)
    md = cuda(m0)
    x = torch.empty((77, 333), dtype=torch.float16, device="cuda")
    norms = torch.empty(1, dtype=torch.float32, device="cuda")
    dm.momentum_normalize(None, [md], [x], norms, beta=0.95, eps=EPS)
    dm.check_status()
    assert torch.equal(md.cpu(), torch.from_numpy(m0))  # untouched
    assert abs(norms.item() - ns64.frobenius_norm(m0)) <= TOL_F32 * ns64.frobenius_norm(m0)


# ------------------------------------------------------------------------------- single-matrix NS


def run_ns(dm, g, coeffs, restarts, backend):
    x = cuda(g.astype(np.float32))
    dm.ns(x, coeffs, restarts, backend, EPS)
    dm.check_status()
    return x.cpu().numpy()


@pytest.mark.parametrize("backend", ["direct", "gram"])
def test_single_matrix_256x1024_you(dm, backend):
    """The small parity case: 256 x 1024 N(0, 1), YOU coefficients, restart [2] for Gram."""
    g = workloads.gaussian((256, 1024), 1.0, 1)
    got = run_ns(dm, g, dm.YOU, (2,), backend)
    want = ns64.newton_schulz(g, ns64.YOU, (2,), backend, EPS)
    assert rel(got, want) <= TOL_NS


@pytest.mark.parametrize("backend", ["direct", "gram"])
@pytest.mark.parametrize("shape", [(300, 1000), (1000, 300), (129, 257), (100, 100), (1, 7), (7, 1), (640, 640),
                                   (33, 2000)])
def test_ns_ragged_shapes(dm, backend, shape):
    g = workloads.gaussian(shape, 1.0, sum(shape))
    got = run_ns(dm, g, dm.YOU, (2,), backend)
    want = ns64.newton_schulz(g, ns64.YOU, (2,), backend, EPS)
    assert rel(got, want) <= TOL_NS


@pytest.mark.parametrize("restarts", [(), (1, 3), (0,), (1, 2, 3, 4)])
def test_gram_restart_lists(dm, restarts):
    g = workloads.gaussian((200, 600), 1.0, 9)
    got = run_ns(dm, g, dm.YOU, restarts, "gram")
    want = ns64.newton_schulz(g, ns64.YOU, restarts, "gram", EPS)
    assert rel(got, want) <= TOL_NS


def test_custom_steps_and_identity_polynomial(dm):
    g = workloads.gaussian((96, 160), 1.0, 10)
    x, _ = ns64.normalise(g, EPS)
    got = run_ns(dm, g, ((1.0, 0.0, 0.0),) * 3, (1,), "gram")
    assert rel(got, x) <= TOL_X * 4
    cubic = ((1.5, -0.5, 0.0),) * 7
    for backend in ("direct", "gram"):
        got = run_ns(dm, g, cubic, (2, 5), backend)
        assert rel(got, ns64.newton_schulz(g, cubic, (2, 5), backend, EPS)) <= TOL_NS


def test_zero_matrix_gives_zero(dm):
    for backend in ("direct", "gram"):
        got = run_ns(dm, np.zeros((64, 200), np.float32), dm.POLAR_EXPRESS, (2,), backend)
        assert not np.any(got)


def test_overflow_is_reported(dm):
    """A rank-1 input has its only normalised singular value at 1, where the printed POLAR_EXPRESS
    polynomials grow past the fp16 range: the run must report NONFINITE, not return silently."""
    u = workloads.gaussian((64, 1), 1.0, 11)
    v = workloads.gaussian((1, 256), 1.0, 12)
    x = cuda((u @ v).astype(np.float32))
    dm.ns(x, dm.POLAR_EXPRESS, (2,), "gram", EPS)
    with pytest.raises(dm.DmuonError) as ei:
        dm.check_status()
    assert ei.value.status == dm.ERR_NONFINITE
    dm.check_status()  # the word was cleared


def test_ns_deterministic(dm):
    g = workloads.gaussian((384, 1536), 1.0, 13)
    a = run_ns(dm, g, dm.POLAR_EXPRESS, (2,), "gram")
    b = run_ns(dm, g, dm.POLAR_EXPRESS, (2,), "gram")
    assert np.array_equal(a, b)


def test_auto_backend_picks_per_matrix(dm):
    """auto runs direct where it needs fewer flops (n < 4m/3: square-ish) and Gram elsewhere, in the same
    grouped launches; each matrix must match the oracle for the form it ran."""
    shapes = [(384, 384), (256, 1024), (1024, 300), (500, 600), (96, 520), (640, 640)]
    W = [workloads.gaussian(s, 0.02, 700 + i) for i, s in enumerate(shapes)]
    G = [workloads.gaussian(s, 1.0, 800 + i) for i, s in enumerate(shapes)]
    Wd = [cuda(w) for w in W]
    Md = [torch.zeros(s, dtype=torch.float32, device="cuda") for s in shapes]
    dm.muon_step(Wd, [cuda(g) for g in G], Md, lr=0.02, beta=0.95, coeffs=dm.YOU, restarts=(2,), backend="auto")
    dm.check_status()
    for i, s in enumerate(shapes):
        form = "direct" if dm.auto_uses_direct(*s) else "gram"
        ref = muon_ref(W[i], G[i], np.zeros(s), 0.02, 0.95, ns64.YOU, (2,), form)
        assert check_update(W[i], Wd[i].cpu().numpy(), ref, 0.02) <= TOL_NS, (s, form)
    assert dm.auto_uses_direct(384, 384) and dm.auto_uses_direct(500, 600)
    assert not dm.auto_uses_direct(256, 1024) and not dm.auto_uses_direct(1024, 300)


# ------------------------------------------------------------------------------- closed-form matrices


@pytest.mark.slow
@pytest.mark.parametrize("case", ["square_log_uniform", "top_tenth"])
@pytest.mark.parametrize("backend", ["gram", "direct"])
def test_closed_form_full_size(dm, case, backend):
    """4096 x 4096 with log-uniform spectrum in [1e-6, 1], and 2048 x 8192 with 205 singular values at 1
    and the rest at 1e-4; POLAR_EXPRESS coefficients; same fp32 input on both sides."""
    if case == "square_log_uniform":
        sigma = workloads.log_uniform_spectrum(4096, 1e-6, 1.0, 2)
        x, _, _ = workloads.closed_form_matrix(4096, 4096, sigma, 2)
    else:
        sigma = workloads.top_fraction_spectrum(2048, 0.1, 1.0, 1e-4)
        x, _, _ = workloads.closed_form_matrix(2048, 8192, sigma, 3)
    g = x.astype(np.float32)
    got = run_ns(dm, g, dm.POLAR_EXPRESS, (2,), backend)
    want = ns64.newton_schulz(g, ns64.POLAR_EXPRESS, (2,), backend, EPS)
    assert rel(got, want) <= TOL_NS


# ------------------------------------------------------------------------------- Muon step


def muon_ref(w0, g, m0, lr, beta, coeffs, restarts, backend):
    return ns64.muon_step(w0, g, m0, lr, beta, coeffs, restarts, backend, EPS)


def check_update(w0, w_gpu, ref, lr):
    upd = (np.asarray(w0, np.float64) - np.asarray(w_gpu, np.float64)) / lr
    return rel(upd, ref["O"])


@pytest.mark.parametrize("backend", ["gram", "direct"])
def test_muon_step_two_steps(dm, backend):
    """Two consecutive steps from a zero momentum (the second exercises beta), mixed orientations."""
    shapes = [(256, 1024), (1024, 256), (200, 200), (96, 520)]
    W = [workloads.gaussian(s, 0.02, 70 + i) for i, s in enumerate(shapes)]
    G1 = [workloads.gaussian(s, 1.0, 80 + i) for i, s in enumerate(shapes)]
    G2 = [workloads.gaussian(s, 1.0, 90 + i) for i, s in enumerate(shapes)]
    Wd = [cuda(w) for w in W]
    Md = [torch.zeros(s, dtype=torch.float32, device="cuda") for s in shapes]
    norms = torch.empty(len(shapes), dtype=torch.float32, device="cuda")
    Mh = [np.zeros(s) for s in shapes]
    Wh = [w.astype(np.float64) for w in W]
    for G in (G1, G2):
        w_before = [wd.cpu().numpy().astype(np.float64) for wd in Wd]
        Gd = [cuda(g) for g in G]
        dm.muon_step(Wd, Gd, Md, lr=0.02, beta=0.95, coeffs=dm.YOU, restarts=(2,), backend=backend,
                     norms_out=norms)
        dm.check_status()
        nh = norms.cpu().numpy()
        for i in range(len(shapes)):
            ref = muon_ref(w_before[i], G[i], Mh[i], 0.02, 0.95, ns64.YOU, (2,), backend)
            assert rel(Md[i].cpu().numpy(), ref["M"]) <= TOL_F32
            assert abs(nh[i] - ref["norm"]) <= TOL_F32 * ref["norm"]
            assert check_update(w_before[i], Wd[i].cpu().numpy(), ref, 0.02) <= TOL_NS
            Mh[i] = Md[i].cpu().numpy().astype(np.float64)
            Wh[i] = ref["W"]


def test_prepared_step_matches_one_shot_call(dm):
    """MuonStep (pointers marshalled once) must give bit-identical results to muon_step."""
    shapes = [(96, 520), (520, 96), (200, 200)]
    W = [workloads.gaussian(s, 0.02, 900 + i) for i, s in enumerate(shapes)]
    G = [workloads.gaussian(s, 1.0, 910 + i) for i, s in enumerate(shapes)]
    runs = []
    for prepared in (False, True):
        Wd = [cuda(w) for w in W]
        Gd = [cuda(g) for g in G]
        Md = [torch.zeros(s, dtype=torch.float32, device="cuda") for s in shapes]
        if prepared:
            step = dm.MuonStep(Wd, Gd, Md, coeffs=dm.POLAR_EXPRESS, restarts=(2,), backend="gram")
            step(lr=0.02, beta=0.95)
            step(lr=0.02, beta=0.95)
        else:
            for _ in range(2):
                dm.muon_step(Wd, Gd, Md, lr=0.02, beta=0.95, coeffs=dm.POLAR_EXPRESS, restarts=(2,), backend="gram")
        dm.check_status()
        runs.append([w.cpu() for w in Wd] + [m.cpu() for m in Md])
    assert all(torch.equal(a, b) for a, b in zip(*runs))


SMALL_SHAPES = [(128, 512), (512, 128), (100, 300), (300, 100), (1, 7), (7, 1), (64, 64), (128, 128), (17, 500),
                (128, 130), (33, 5)]


@pytest.mark.parametrize("backend,restarts", [("gram", (2,)), ("gram", (1, 3)), ("direct", ()), ("auto", (2,))])
def test_small_fused_kernel_matches_oracle(dm, backend, restarts):
    """Every matrix with m <= 128 and n <= 512: the whole iteration runs in one fused launch (including W
    rows that are not 16-byte aligned, written directly instead of by TMA)."""
    W = [workloads.gaussian(s, 0.02, 1100 + i) for i, s in enumerate(SMALL_SHAPES)]
    G = [workloads.gaussian(s, 1.0, 1200 + i) for i, s in enumerate(SMALL_SHAPES)]
    Wd = [cuda(w) for w in W]
    Md = [torch.zeros(s, dtype=torch.float32, device="cuda") for s in SMALL_SHAPES]
    dm.timing_enable(True)
    dm.muon_step(Wd, [cuda(g) for g in G], Md, lr=0.02, beta=0.95, coeffs=dm.YOU, restarts=restarts,
                 backend=backend)
    t = dm.timing_read()
    dm.timing_enable(False)
    dm.check_status()
    assert t["gemm_tc"][1] == 1  # one launch for the whole Newton-Schulz part
    for i, s in enumerate(SMALL_SHAPES):
        form = backend if backend != "auto" else ("direct" if dm.auto_uses_direct(*s) else "gram")
        ref = muon_ref(W[i], G[i], np.zeros(s), 0.02, 0.95, ns64.YOU, restarts, form)
        assert rel(Md[i].cpu().numpy(), ref["M"]) <= TOL_F32
        assert check_update(W[i], Wd[i].cpu().numpy(), ref, 0.02) <= TOL_NS, (s, form)


@pytest.mark.parametrize("backend,restarts", [("gram", (1, 3)), ("direct", ())])
def test_small_fused_kernel_several_matrices_per_cta(dm, backend, restarts):
    """More small matrices than CTAs (one per SM): each CTA runs two or three in turn, fetching the next
    matrix's X while the current one's weight update drains (Gram) or after it (direct). A sample is
    checked against the oracle; every matrix must be bit-identical to running it alone."""
    shapes = (SMALL_SHAPES * 30)[:320]
    W = [workloads.gaussian(s, 0.02, 2100 + i) for i, s in enumerate(shapes)]
    G = [workloads.gaussian(s, 1.0, 2600 + i) for i, s in enumerate(shapes)]
    Wd = [cuda(w) for w in W]
    Md = [torch.zeros(s, dtype=torch.float32, device="cuda") for s in shapes]
    dm.muon_step(Wd, [cuda(g) for g in G], Md, lr=0.02, beta=0.95, coeffs=dm.YOU, restarts=restarts,
                 backend=backend)
    dm.check_status()
    for i in list(range(0, 320, 23)) + [151, 152, 303, 304, 319]:
        ref = muon_ref(W[i], G[i], np.zeros(shapes[i]), 0.02, 0.95, ns64.YOU, restarts, backend)
        assert check_update(W[i], Wd[i].cpu().numpy(), ref, 0.02) <= TOL_NS, (i, shapes[i])
        alone_w = [cuda(W[i])]
        dm.muon_step(alone_w, [cuda(G[i])], [torch.zeros(shapes[i], dtype=torch.float32, device="cuda")], lr=0.02,
                     beta=0.95, coeffs=dm.YOU, restarts=restarts, backend=backend)
        assert torch.equal(alone_w[0], Wd[i]), (i, shapes[i])
    dm.check_status()


def test_small_fused_ns_in_place(dm):
    for shape in ((128, 512), (512, 128), (1, 1), (96, 160)):
        for backend in ("gram", "direct"):
            g = workloads.gaussian(shape, 1.0, 1300 + sum(shape))
            got = run_ns(dm, g, dm.YOU, (2,), backend)
            assert rel(got, ns64.newton_schulz(g, ns64.YOU, (2,), backend, EPS)) <= TOL_NS


def test_small_matrix_set_one_grouped_step(dm):
    """2048 gradients of 128 x 512 plus 512 of 512 x 128, N(0, 1e-3^2), beta 0.95 from zero, Gram with
    restart [2]: the whole iteration of all 2560 matrices in one fused launch. Graded with YOU at 2e-2. The
    printed POLAR_EXPRESS set is run too and held to 6e-2: on these Gaussian 128 x 512 matrices the
    normalised singular values lie in [0.044, 0.133], where the composition of the printed POLAR_EXPRESS
    polynomials runs from 1.02 up to 2.5e5 with slopes up to 4e7, so fp16 rounding of the intermediates is
    amplified far more than with YOU (range 0.98 .. 1.03, slopes below 12). Any fp16 iteration lands near
    5e-2 here: the fp16 error model (oracle/fp16_model.py) gives 4.7e-2 to 5.6e-2 on these matrices, and
    tests/test_gpu_error_floor.py holds the kernel to that floor matrix by matrix."""
    shapes = workloads.small_set_shapes()
    G = [workloads.gaussian(s, 1e-3, 1000 + i) for i, s in enumerate(shapes)]
    W = [workloads.gaussian(s, 0.02, 5000 + i) for i, s in enumerate(shapes)]
    sample = list(range(0, 2048, 97)) + [2047, 2048, 2300, 2559]
    for coeffs, tol in ((dm.YOU, TOL_NS), (dm.POLAR_EXPRESS, 6e-2)):
        Wd = [cuda(w) for w in W]
        Gd = [cuda(g) for g in G]
        Md = [torch.zeros(s, dtype=torch.float32, device="cuda") for s in shapes]
        dm.muon_step(Wd, Gd, Md, lr=0.02, beta=0.95, coeffs=coeffs, restarts=(2,), backend="gram")
        dm.check_status()
        oc = ns64.YOU if coeffs == dm.YOU else ns64.POLAR_EXPRESS
        for i in sample:
            ref = muon_ref(W[i], G[i], np.zeros(shapes[i]), 0.02, 0.95, oc, (2,), "gram")
            assert rel(Md[i].cpu().numpy(), ref["M"]) <= TOL_F32
            assert check_update(W[i], Wd[i].cpu().numpy(), ref, 0.02) <= tol


def _llama_run(dm, layers, seed, sample_names, backend):
    """Two Muon steps over `layers` Llama-3-8B layers of Muon-target matrices: bf16 grads N(0, 1e-3^2), fp32 W
    N(0, 0.02^2), POLAR_EXPRESS, Gram restart [2]. Step 1 starts from zero momentum; step 2 takes a second
    seeded gradient on top of step 1's momentum, so M <- beta M + G runs with M != 0 through the bulk-copy
    momentum pass at full size. The sampled matrices get host-generated gradients and weights (seeded per
    matrix and step) and are compared with the oracle after each step on M and ||M|| (1e-5) and on the
    update (W_before - W_after) / lr (2e-2), the oracle taking the GPU's W and M from before the step; the
    other matrices are filled on the device and are not compared. The device buffers stay the same across
    the two steps (new gradients are copied into them), as in a training loop."""
    shapes = workloads.llama3_8b_shapes(layers)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    Wd, Gd, Md, host = [], [], [], {}
    for i, (name, r, c) in enumerate(shapes):
        if name in sample_names:
            grads = [workloads.round_to_bf16(workloads.gaussian((r, c), 1e-3, seed * 1000 + 250 * s + i))
                     for s in (0, 2)]
            w = workloads.gaussian((r, c), 0.02, seed * 1000 + 500 + i)
            host[i] = grads
            Gd.append(torch.empty((r, c), dtype=torch.bfloat16, device="cuda"))
            Wd.append(cuda(w))
        else:
            Gd.append(torch.empty((r, c), dtype=torch.bfloat16, device="cuda"))
            Wd.append(torch.randn((r, c), generator=gen, device="cuda") * 0.02)
        Md.append(torch.zeros((r, c), dtype=torch.float32, device="cuda"))
    norms = torch.empty(len(shapes), dtype=torch.float32, device="cuda")
    for step in range(2):
        for i, (name, r, c) in enumerate(shapes):
            if i in host:
                bits = host[i][step][1]
                Gd[i].copy_(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16))
            else:
                Gd[i].copy_((torch.randn((r, c), generator=gen, device="cuda") * 1e-3).to(torch.bfloat16))
        before = {i: (Wd[i].cpu().numpy().astype(np.float64), Md[i].cpu().numpy().astype(np.float64)) for i in host}
        dm.muon_step(Wd, Gd, Md, lr=0.02, beta=0.95, coeffs=dm.POLAR_EXPRESS, restarts=(2,), backend=backend,
                     norms_out=norms)
        dm.check_status()
        nh = norms.cpu().numpy()
        for i, (w0, m0) in before.items():
            if step == 0:
                assert not np.any(m0)
            g = host[i][step][0]
            ref = muon_ref(w0, g, m0, 0.02, 0.95, ns64.POLAR_EXPRESS, (2,), backend)
            where = (shapes[i][0], f"step {step + 1}")
            assert rel(Md[i].cpu().numpy(), ref["M"]) <= TOL_F32, where
            assert abs(nh[i] - ref["norm"]) <= TOL_F32 * ref["norm"], where
            err = check_update(w0, Wd[i].cpu().numpy(), ref, 0.02)
            assert err <= TOL_NS, (where, err)
    del Wd, Gd, Md
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_llama_4_layers(dm):
    names = {"layers.0.q_proj", "layers.1.k_proj", "layers.2.gate_proj", "layers.3.down_proj"}
    _llama_run(dm, 4, 5, names, "gram")


@pytest.mark.slow
@pytest.mark.parametrize("backend", ["gram", "direct"])
def test_llama_whole_model(dm, backend):
    """All 32 layers (224 matrices, 6.98 G parameters) in one call; sampled matrices from the first and
    last layers are compared with the oracle."""
    names = {"layers.0.k_proj", "layers.31.v_proj", "layers.0.o_proj"}
    if backend == "gram":
        names |= {"layers.31.up_proj", "layers.0.down_proj"}
    _llama_run(dm, 32, 6, names, backend)
    dm.release_workspace()


def test_plan_info_and_launch_timing(dm):
    """dmuon_plan_info and the per-launch timing record agree with the plan that ran: the GEMM launches
    counted both ways match, and the executed MMA flops lie between the algorithmic count (symmetric
    products at half) and the dense count padded to whole 256 x 256 tiles and 64-wide K slices."""
    shapes = [(520, 264), (264, 1040), (1024, 256), (300, 300)]
    W = [cuda(workloads.gaussian(s, 0.02, 60 + i)) for i, s in enumerate(shapes)]
    G = [cuda(workloads.gaussian(s, 1.0, 65 + i)) for i, s in enumerate(shapes)]
    M = [torch.zeros(s, dtype=torch.float32, device="cuda") for s in shapes]
    dm.timing_enable(True)
    dm.muon_step(W, G, M, lr=0.02, beta=0.95, coeffs=dm.YOU, restarts=(2,), backend="gram")
    rec = dm.timing_read_launches()
    dm.timing_enable(False)
    dm.check_status()
    flops, tiles, gemm_launches = dm.plan_info()
    assert sum(1 for c, _ in rec if c == "gemm_tc") == gemm_launches > 0
    assert [c for c, _ in rec[:3]] == ["momentum_sumsq", "finalize_norms", "normalize_cast"]
    assert all(ms >= 0 for _, ms in rec)
    algo = sum(dm.gram_flops(r, c) for r, c in shapes)
    padded = sum(dm.gram_flops(-(-min(r, c) // 256) * 256, -(-max(r, c) // 256) * 256, dense=True)
                 for r, c in shapes)
    assert tiles > 0 and algo <= flops <= padded


def test_small_launches_take_128x64_tiles(dm):
    """A lone 256 x 1024 matrix: every GEMM launch would fill under half the SMs with 128 x 128 tiles, so
    each takes 128 x 64 tiles. 17 launches (Gram, restart [2]); the products of m <= 256 are computed in
    full: 8 tiles for each 256 x 256 product, 16 for the launch holding two of them, 32 for each Q X
    (256 x 1024). Executed flops: 2 * 128 * 64 * K per tile (K = 1024 for X X^T, 256 otherwise)."""
    W = [cuda(workloads.gaussian((256, 1024), 0.02, 70))]
    G = [cuda(workloads.gaussian((256, 1024), 1.0, 71))]
    M = [torch.zeros((256, 1024), dtype=torch.float32, device="cuda")]
    dm.muon_step(W, G, M, lr=0.02, beta=0.95, coeffs=dm.YOU, restarts=(2,), backend="gram")
    dm.check_status()
    flops, tiles, gemm_launches = dm.plan_info()
    assert gemm_launches == 17
    assert tiles == 14 * 8 + 16 + 2 * 32
    assert flops == 2.0 * 128 * 64 * (2 * 8 * 1024 + (12 * 8 + 16 + 2 * 32) * 256)


@pytest.mark.parametrize("shape", [(1, 1 << 20), (1 << 20, 1), (8, 1 << 18), (3, 100003)])
@pytest.mark.parametrize("backend", ["gram", "direct"])
def test_extreme_aspect_ratios(dm, shape, backend):
    """Very long rows (m up to 8 after orientation, n up to 2^20): the Gram matrix is tiny while X X^T and
    Q X run over a long K or N; a prime-length side leaves a ragged tail in every tile row."""
    g = workloads.gaussian(shape, 1.0, 31 + shape[0])
    got = run_ns(dm, g, dm.YOU, (2,), backend)
    want = ns64.newton_schulz(g, ns64.YOU, (2,), backend, EPS)
    assert rel(got, want) <= TOL_NS


def test_nonfinite_gradient_is_reported_and_others_unaffected(dm):
    """An inf in one matrix's gradient makes that matrix's norm and X non-finite: the step reports NONFINITE
    instead of returning silently. The other matrices of the call are computed as usual."""
    shapes = [(256, 1024), (300, 700)]
    W = [workloads.gaussian(s, 0.02, 1700 + i) for i, s in enumerate(shapes)]
    G = [workloads.gaussian(s, 1.0, 1800 + i) for i, s in enumerate(shapes)]
    bad = G[0].copy()
    bad[5, 7] = np.inf
    Wd = [cuda(w) for w in W]
    Md = [torch.zeros(s, dtype=torch.float32, device="cuda") for s in shapes]
    dm.muon_step(Wd, [cuda(bad), cuda(G[1])], Md, lr=0.02, beta=0.95, coeffs=dm.YOU, restarts=(2,), backend="gram")
    with pytest.raises(dm.DmuonError) as ei:
        dm.check_status()
    assert ei.value.status == dm.ERR_NONFINITE
    ref = muon_ref(W[1], G[1], np.zeros(shapes[1]), 0.02, 0.95, ns64.YOU, (2,), "gram")
    assert check_update(W[1], Wd[1].cpu().numpy(), ref, 0.02) <= TOL_NS
    dm.check_status()  # cleared
