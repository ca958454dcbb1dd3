"""Input generators: determinism, shapes, and the bf16 rounding against torch's own conversion."""

import numpy as np
import torch

import workloads


def test_gaussian_is_seeded():
    a = workloads.gaussian((3, 5), 1e-3, 7)
    b = workloads.gaussian((3, 5), 1e-3, 7)
    assert a.dtype == np.float32 and np.array_equal(a, b)
    assert not np.array_equal(a, workloads.gaussian((3, 5), 1e-3, 8))


def test_bf16_rounding_matches_torch():
    x = workloads.gaussian((4096,), 1.0, 3) * np.float32(1e-3)
    vals, bits = workloads.round_to_bf16(x)
    t = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(t.float().numpy(), vals)
    assert np.array_equal(t.view(torch.int16).numpy().view(np.uint16), bits)


def test_shape_sets():
    s = workloads.llama3_8b_shapes(32)
    assert len(s) == 224
    assert sum(r * c for _, r, c in s) == 6_979_321_856
    small = workloads.small_set_shapes()
    assert len(small) == 2560 and small[0] == (128, 512) and small[-1] == (512, 128)


def test_closed_form_matrix_has_prescribed_spectrum():
    sig = workloads.log_uniform_spectrum(16, 1e-6, 1.0, 2)
    x, u, v = workloads.closed_form_matrix(16, 40, sig, 2)
    assert np.allclose(np.linalg.svd(x, compute_uv=False), sig, rtol=1e-9, atol=1e-15)
    top = workloads.top_fraction_spectrum(2048, 0.1, 1.0, 1e-4)
    assert int((top == 1.0).sum()) == 205
