"""GPU: the checked build (libdmuon_checked.so: device-side range checks compiled in, the debugging stand-in
for a memory checker).

In a child process that loads the checked library: its range self-test launches one GEMM whose only tile
lies outside its product, and the next status check reports DMUON_ERR_RANGE (the tile is skipped before
anything is read or written); then every kind of launch -- the row-wise passes, grouped GEMM phases with
symmetric and full products on CTA pairs and single CTAs, the fused small-matrix kernel, the column-split
Gram form, AdamW and the allocation-free entry -- runs with no range failure. The child saves its results;
the same calls through the regular library in this process must give the same bits (the checks change
no arithmetic)."""

import os
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run_all(dm):
    """The same calls in either build; returns {name: numpy array}."""
    out = {}
    shapes = [(256, 1024), (1024, 300), (520, 264), (96, 520)]
    W = [torch.from_numpy(workloads.gaussian(s, 0.02, 10 + i)).cuda() for i, s in enumerate(shapes)]
    G = [torch.from_numpy(workloads.gaussian(s, 1.0, 20 + i)).cuda() for i, s in enumerate(shapes)]
    M = [torch.zeros(s, device="cuda") for s in shapes]
    for backend in ("gram", "direct"):
        dm.muon_step(W, G, M, lr=0.02, beta=0.95, coeffs=dm.YOU, restarts=(2,), backend=backend)
        dm.check_status()
    out.update({f"W{i}": w for i, w in enumerate(W)})
    out.update({f"M{i}": m for i, m in enumerate(M)})
    small = [(128, 512), (512, 128), (7, 1)]
    Ws = [torch.from_numpy(workloads.gaussian(s, 0.02, 30 + i)).cuda() for i, s in enumerate(small)]
    dm.muon_step(Ws, [torch.from_numpy(workloads.gaussian(s, 1.0, 40 + i)).cuda() for i, s in enumerate(small)],
                 [torch.zeros(s, device="cuda") for s in small], lr=0.02, beta=0.95, coeffs=dm.YOU)
    dm.check_status()
    out.update({f"Ws{i}": w for i, w in enumerate(Ws)})
    x = torch.from_numpy(workloads.gaussian((192, 2048), 1.0, 50)).cuda()
    dm.ns_tp(x, 4, dm.POLAR_EXPRESS, (2,))
    dm.check_status()
    out["tp"] = x
    p = [torch.from_numpy(workloads.gaussian((5000,), 0.02, 60)).cuda()]
    g = [torch.from_numpy(workloads.gaussian((5000,), 1e-3, 61)).cuda()]
    m, v = [torch.zeros(5000, device="cuda")], [torch.zeros(5000, device="cuda")]
    dm.adamw_step(p, g, m, v, step=1)
    dm.check_status()
    out["adam"] = p[0]
    mo = torch.from_numpy(workloads.gaussian((300, 700), 1e-3, 70)).cuda()
    xo = torch.empty((300, 700), dtype=torch.float16, device="cuda")
    n = torch.empty(1, device="cuda")
    dm.momentum_normalize_noalloc(torch.from_numpy(workloads.gaussian((300, 700), 1e-3, 71)).cuda(), mo, xo, n)
    dm.check_status()
    out["noalloc_x"] = xo.float()
    out["noalloc_norm"] = n
    return {k: t.cpu().numpy() for k, t in out.items()}


CHILD = r"""
import os, sys
sys.path.insert(0, {root!r})
import numpy as np
import torch
import newton_schulz_momentum_gb300 as dm
assert "range checks" in dm.version(), dm.version()
dm.selftest_range_check()
try:
    dm.check_status()
    raise SystemExit("the range self-test was not reported")
except dm.DmuonError as e:
    assert e.status == dm.ERR_RANGE, e
dm.check_status()  # cleared
sys.path.insert(0, os.path.join({root!r}, "tests"))
from test_gpu_checked_build import _run_all
np.savez({out!r}, **_run_all(dm))
print("checked build ok")
"""


def test_checked_build_reports_a_planted_range_failure_and_nothing_else(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_momentum_gb300 as dm
    out = str(tmp_path / "checked.npz")
    env = dict(os.environ, DMUON_LIBRARY="checked")
    proc = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, out=out)], env=env, capture_output=True,
                          text=True, timeout=600)
    assert proc.returncode == 0, proc.stdout + proc.stderr
    checked = np.load(out)
    regular = _run_all(dm)
    assert sorted(checked.files) == sorted(regular)
    for k in regular:
        assert np.array_equal(checked[k], regular[k]), k
