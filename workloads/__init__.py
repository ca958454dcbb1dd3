"""Seeded synthetic inputs for the owner-rank Muon update.

This module holds input generation only -- no step of the method. Both the CUDA path's tests and
benchmark and the CPU oracle's tests draw their inputs from here, so the two sides see the same
bytes. Everything is NumPy on the host, seeded with ``numpy.random.default_rng``.

Workloads (shapes and distributions; nothing is read from a dataset or a checkpoint):

* single matrix 256 x 1024, G ~ N(0, 1) fp32 (small parity case);
* closed-form matrices X = U diag(s) V^T, U and V from QR of seeded Gaussians:
  4096 x 4096 with s log-uniform in [1e-6, 1], and 2048 x 8192 with the top 10% of s at 1 and the
  rest at 1e-4;
* many small matrices: 2048 of 128 x 512 and 512 of 512 x 128, G ~ N(0, 1e-3^2) fp32;
* the Muon-target matrices of a Llama-3-8B-shaped model (h 4096, ffn 14336, GQA kv 1024), per layer
  q/o 4096 x 4096, k/v 1024 x 4096, gate/up 14336 x 4096, down 4096 x 14336 (rows x cols as
  stored, out x in), bf16 gradients N(0, 1e-3^2), fp32 weights N(0, 0.02^2).
"""

from __future__ import annotations

import numpy as np

LLAMA3_8B_LAYER = (
    ("q_proj", 4096, 4096),
    ("k_proj", 1024, 4096),
    ("v_proj", 1024, 4096),
    ("o_proj", 4096, 4096),
    ("gate_proj", 14336, 4096),
    ("up_proj", 14336, 4096),
    ("down_proj", 4096, 14336),
)


def llama3_8b_non_muon_numels():
    """[(name, numel)] of the Llama-3-8B parameters that are not Muon targets (AdamW's share): token
    embeddings and the untied output head (vocabulary 128256 x 4096) and the 65 RMSNorm weights (4096)."""
    out = [("embed_tokens", 128256 * 4096), ("lm_head", 128256 * 4096), ("norm", 4096)]
    for i in range(32):
        out += [(f"layers.{i}.input_layernorm", 4096), (f"layers.{i}.post_attention_layernorm", 4096)]
    return out


def llama3_8b_shapes(layers):
    """[(name, rows, cols)] for `layers` decoder layers (32 for the whole model: 224 matrices)."""
    return [(f"layers.{i}.{name}", r, c) for i in range(layers) for name, r, c in LLAMA3_8B_LAYER]


def small_set_shapes():
    """2048 matrices of 128 x 512 followed by 512 of 512 x 128."""
    return [(128, 512)] * 2048 + [(512, 128)] * 512


def gaussian(shape, std, seed):
    """float32 array of N(0, std^2) draws from default_rng(seed)."""
    rng = np.random.default_rng(seed)
    out = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def round_to_bf16(x):
    """Round float32 values to the nearest bfloat16 (ties to even); returns (values as float32, raw
    uint16 bit patterns). NaN/Inf are not expected in these workloads."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32), (r >> np.uint32(16)).astype(np.uint16)


def random_orthogonal(rng, n, k=None):
    """n x k matrix with orthonormal columns (QR of a Gaussian, column signs fixed by diag(R))."""
    k = n if k is None else k
    q, r = np.linalg.qr(rng.standard_normal((n, k)))
    return q * np.sign(np.diag(r))


def closed_form_matrix(m, n, sigma, seed):
    """X = U diag(sigma) V^T in float64 with U (m x k), V (n x k) orthonormal, k = min(m, n).
    Returns (X, U, V)."""
    rng = np.random.default_rng(seed)
    k = min(m, n)
    u = random_orthogonal(rng, m, k)
    v = random_orthogonal(rng, n, k)
    return (u * np.asarray(sigma, dtype=np.float64)) @ v.T, u, v


def log_uniform_spectrum(k, lo, hi, seed):
    """k values log-uniform in [lo, hi], sorted descending."""
    rng = np.random.default_rng(seed)
    return np.sort(10.0 ** rng.uniform(np.log10(lo), np.log10(hi), size=k))[::-1].copy()


def top_fraction_spectrum(k, frac, top, rest):
    """round(frac * k) values equal to `top`, the others equal to `rest`."""
    s = np.full(k, rest, dtype=np.float64)
    s[: int(round(frac * k))] = top
    return s
