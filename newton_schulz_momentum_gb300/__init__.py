"""Thin Python binding of libdmuon (the C ABI in include/dmuon.h): argument marshalling only.

Every step of the update runs in the CUDA library; this module passes device pointers, sizes and the
current CUDA stream through ctypes. There is no CPU fallback: if libdmuon.so has not been built, every
call raises ``LibraryNotBuilt``.

    import newton_schulz_momentum_gb300 as dm
    dm.ns(x, dm.POLAR_EXPRESS, restarts=(2,), backend="gram")          # in place, fp32 CUDA tensor
    dm.muon_step(params, grads, momenta, lr=0.02, beta=0.95, coeffs=dm.POLAR_EXPRESS)

The pages' own names -- newton_schulz, NewtonSchulz and the Muon optimizer -- live in
newton_schulz_momentum_gb300.optim (imports torch) and are reachable here as attributes.
"""

from __future__ import annotations

import ctypes
import os
from typing import Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
# DMUON_LIBRARY=checked loads the build with device-side range checks (libdmuon_checked.so) instead.
LIB_PATH = os.path.join(_HERE, "libdmuon_checked.so" if os.environ.get("DMUON_LIBRARY") == "checked"
                        else "libdmuon.so")
CHECKED_LIB_PATH = os.path.join(_HERE, "libdmuon_checked.so")

# Coefficient tables printed on the DMuon "Newton-Schulz 变体" page, section "系数集".
POLAR_EXPRESS = (
    (7.893, -20.381, 14.939),
    (3.912, -2.544, 0.470),
    (3.761, -2.512, 0.476),
    (3.160, -2.148, 0.440),
    (2.191, -1.441, 0.361),
)
YOU = (
    (4.0848, -6.8946, 2.9270),
    (3.9505, -6.3029, 2.6377),
    (3.7418, -5.5913, 2.3037),
    (2.8769, -3.1427, 1.2046),
    (2.8366, -3.0525, 1.2012),
)
DEFAULT_RESTARTS = (2,)

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_OOM, ERR_CUDA, ERR_TIMEOUT, ERR_NONFINITE, ERR_RANGE = range(8)
_STATUS_NAMES = {1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "OOM", 4: "CUDA", 5: "TIMEOUT", 6: "NONFINITE", 7: "RANGE"}
BACKENDS = {"direct": 0, "gram": 1, "auto": 2}
F32, BF16 = 0, 1

EXPORTS = (
    "dmuon_ns", "dmuon_muon_step", "dmuon_momentum_normalize", "dmuon_gemm_f16", "dmuon_check_status",
    "dmuon_last_error", "dmuon_version", "dmuon_set_workspace_limit", "dmuon_workspace_size",
    "dmuon_release_workspace", "dmuon_timing_enable", "dmuon_timing_read", "dmuon_momentum_normalize_noalloc",
    "dmuon_assign_owners", "dmuon_adamw_step", "dmuon_ns_tp", "dmuon_muon_step_host",
    "dmuon_timing_read_launches", "dmuon_plan_info", "dmuon_selftest_bounded_wait", "dmuon_selftest_range_check",
    "dmuon_set_graph_replay",
)
COST_MODELS = {"elements": 0, "gram_flops": 1, "direct_flops": 2}
NOALLOC_MAX_ELEMS = 268435456
TIMING_CLASSES = ("momentum_sumsq", "finalize_norms", "normalize_cast", "gemm_tc", "adamw", "tp_reduce")


class LibraryNotBuilt(RuntimeError):
    pass


class DmuonError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"dmuon error {_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None

_c_i64p = ctypes.POINTER(ctypes.c_int64)
_c_vpp = ctypes.POINTER(ctypes.c_void_p)
_c_fp = ctypes.POINTER(ctypes.c_float)
_c_ip = ctypes.POINTER(ctypes.c_int)


def lib():
    """Load libdmuon.so (once). Raises LibraryNotBuilt when it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise LibraryNotBuilt(f"{LIB_PATH} is missing; build it with newton_schulz_momentum_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    L.dmuon_ns.argtypes = [vp, i64, i64, _c_fp, i32, _c_ip, i32, i32, f32, vp]
    L.dmuon_ns_tp.argtypes = [vp, i64, i64, i32, _c_fp, i32, _c_ip, i32, f32, vp]
    L.dmuon_muon_step.argtypes = [i32, _c_vpp, _c_vpp, i32, _c_vpp, _c_i64p, _c_i64p, vp, f32, f32, _c_fp, i32,
                                  _c_ip, i32, i32, f32, vp]
    L.dmuon_muon_step_host.argtypes = [i32, _c_vpp, _c_vpp, _c_vpp, i32, _c_vpp, _c_i64p, _c_i64p, vp, f32, f32,
                                       _c_fp, i32, _c_ip, i32, i32, f32, i32, vp]
    L.dmuon_momentum_normalize.argtypes = [i32, _c_vpp, i32, _c_vpp, _c_i64p, _c_i64p, _c_vpp, vp, f32, f32, vp]
    L.dmuon_gemm_f16.argtypes = [i64, i64, i64, vp, i64, vp, i64, i32, vp, i64, vp, i64, f32, f32, f32, i32, vp]
    L.dmuon_check_status.argtypes = [vp]
    L.dmuon_last_error.restype = ctypes.c_char_p
    L.dmuon_version.restype = ctypes.c_char_p
    L.dmuon_set_workspace_limit.argtypes = [ctypes.c_size_t]
    L.dmuon_workspace_size.argtypes = [i32, _c_i64p, _c_i64p, i32, ctypes.POINTER(ctypes.c_size_t)]
    L.dmuon_momentum_normalize_noalloc.argtypes = [vp, i32, vp, i64, i64, vp, vp, f32, f32, vp]
    L.dmuon_timing_enable.argtypes = [i32]
    L.dmuon_set_graph_replay.argtypes = [i32]
    f64 = ctypes.c_double
    L.dmuon_adamw_step.argtypes = [i32, _c_vpp, _c_vpp, i32, _c_vpp, _c_vpp, _c_i64p, f64, f64, f64, f64, f64, i32, vp]
    L.dmuon_assign_owners.argtypes = [i32, _c_i64p, _c_i64p, _c_ip, i32, i32, _c_ip, ctypes.POINTER(ctypes.c_double)]
    L.dmuon_timing_read.argtypes = [ctypes.POINTER(ctypes.c_double), _c_i64p]
    L.dmuon_timing_read_launches.argtypes = [i32, ctypes.POINTER(ctypes.c_double), _c_ip, _c_ip]
    L.dmuon_plan_info.argtypes = [ctypes.POINTER(ctypes.c_double), _c_i64p, _c_ip]
    L.dmuon_selftest_bounded_wait.argtypes = [i64, vp]
    L.dmuon_selftest_range_check.argtypes = [vp]
    for name in EXPORTS:
        if name not in ("dmuon_last_error", "dmuon_version"):
            getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _check(status):
    if status != OK:
        raise DmuonError(status, lib().dmuon_last_error().decode(errors="replace"))


def _ptr(t):
    """Device address of a torch tensor (or an int address, or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _coeff_array(coeffs):
    flat = [float(v) for triple in coeffs for v in triple]
    if len(flat) % 3 or not flat:
        raise ValueError("coeffs must be a non-empty sequence of (a, b, c) triples")
    return (ctypes.c_float * len(flat))(*flat), len(flat) // 3


def _int_array(vals):
    vals = [int(v) for v in vals]
    return (ctypes.c_int * max(len(vals), 1))(*vals), len(vals)


def _backend(backend):
    if isinstance(backend, int):
        return backend
    return BACKENDS[backend]


def version():
    return lib().dmuon_version().decode()


def ns(x, coeffs=POLAR_EXPRESS, restarts=DEFAULT_RESTARTS, backend="gram", eps=1e-7, stream=None):
    """In-place Newton-Schulz of one fp32 CUDA matrix x (rows x cols, contiguous). Returns x."""
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D tensor")
    c, steps = _coeff_array(coeffs)
    r, nr = _int_array(restarts)
    _check(lib().dmuon_ns(_ptr(x), x.shape[0], x.shape[1], c, steps, r, nr, _backend(backend), float(eps),
                          _stream(stream)))
    return x


def ns_tp(x, shards, coeffs=POLAR_EXPRESS, restarts=DEFAULT_RESTARTS, eps=1e-7, stream=None):
    """ns (Gram form) as `shards` tensor-parallel ranks would compute it: per-shard sums of squares and
    per-shard fp32 Gram matrices reduced in a fixed order. In place on an fp32 CUDA matrix; returns x."""
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D tensor")
    c, steps = _coeff_array(coeffs)
    r, nr = _int_array(restarts)
    _check(lib().dmuon_ns_tp(_ptr(x), x.shape[0], x.shape[1], int(shards), c, steps, r, nr, float(eps),
                             _stream(stream)))
    return x


def shard_bounds(long_side, shards):
    """Boundaries ns_tp uses along the long side: t * long_side / shards rounded down to a multiple of 8."""
    return [(t * long_side // shards) // 8 * 8 for t in range(shards)] + [long_side]


def _grad_dtype(grads):
    import torch
    dts = {g.dtype for g in grads}
    if dts == {torch.float32}:
        return F32
    if dts == {torch.bfloat16}:
        return BF16
    raise ValueError("grads must all be float32 or all bfloat16")


def muon_step(params: Sequence, grads: Sequence, momenta: Sequence, lr=0.02, beta=0.95, coeffs=POLAR_EXPRESS,
              restarts=DEFAULT_RESTARTS, backend="gram", eps=1e-7, norms_out=None, stream=None):
    """One batched owner-rank Muon update: M <- beta M + G; W <- W - lr NS(M / (||M|| + eps))."""
    n = len(params)
    if not (len(grads) == len(momenta) == n) or n == 0:
        raise ValueError("params, grads and momenta must be non-empty lists of equal length")
    for w, g, m in zip(params, grads, momenta):
        if w.shape != g.shape or w.shape != m.shape or w.dim() != 2:
            raise ValueError("each param, grad and momentum must be a 2-D tensor of the same shape")
        if not (w.is_contiguous() and g.is_contiguous() and m.is_contiguous()):
            raise ValueError("tensors must be contiguous")
    c, steps = _coeff_array(coeffs)
    r, nr = _int_array(restarts)
    P = (ctypes.c_void_p * n)(*[_ptr(t) for t in params])
    G = (ctypes.c_void_p * n)(*[_ptr(t) for t in grads])
    M = (ctypes.c_void_p * n)(*[_ptr(t) for t in momenta])
    rows = (ctypes.c_int64 * n)(*[t.shape[0] for t in params])
    cols = (ctypes.c_int64 * n)(*[t.shape[1] for t in params])
    _check(lib().dmuon_muon_step(n, P, G, _grad_dtype(grads), M, rows, cols, _ptr(norms_out), float(lr),
                                 float(beta), c, steps, r, nr, _backend(backend), float(eps), _stream(stream)))


class MuonStep:
    """A prepared dmuon_muon_step over fixed tensors: validation and pointer marshalling happen once, so
    each step() is one C call (what a training loop does every iteration with the same buffers).

        step = MuonStep(params, grads, momenta, coeffs=POLAR_EXPRESS, restarts=(2,), backend="gram")
        step(lr=0.02, beta=0.95)          # enqueued on the current CUDA stream

    With host_grads (CPU tensors shaped like grads, ideally pinned) each call is one
    dmuon_muon_step_host: the gradients are copied from host_grads into grads inside the call, in
    `groups` pipelined groups (0: the library chooses) whose copies overlap the computation. Many small
    matrices (64 or more averaging under 4 MiB) are instead gathered by one kernel that reads host memory
    directly, followed by the step as one group.
    """

    def __init__(self, params, grads, momenta, coeffs=POLAR_EXPRESS, restarts=DEFAULT_RESTARTS, backend="gram",
                 eps=1e-7, norms_out=None, host_grads=None, groups=0):
        n = len(params)
        if not (len(grads) == len(momenta) == n) or n == 0:
            raise ValueError("params, grads and momenta must be non-empty lists of equal length")
        for w, g, m in zip(params, grads, momenta):
            if w.shape != g.shape or w.shape != m.shape or w.dim() != 2:
                raise ValueError("each param, grad and momentum must be a 2-D tensor of the same shape")
            if not (w.is_contiguous() and g.is_contiguous() and m.is_contiguous()):
                raise ValueError("tensors must be contiguous")
        self._keep = (list(params), list(grads), list(momenta), norms_out)  # keep the buffers alive
        self._n = n
        self._P = (ctypes.c_void_p * n)(*[_ptr(t) for t in params])
        self._G = (ctypes.c_void_p * n)(*[_ptr(t) for t in grads])
        self._M = (ctypes.c_void_p * n)(*[_ptr(t) for t in momenta])
        self._rows = (ctypes.c_int64 * n)(*[t.shape[0] for t in params])
        self._cols = (ctypes.c_int64 * n)(*[t.shape[1] for t in params])
        self._gdtype = _grad_dtype(grads)
        self._coeffs, self._steps = _coeff_array(coeffs)
        self._restarts, self._nr = _int_array(restarts)
        self._backend = _backend(backend)
        self._eps = float(eps)
        self._norms = _ptr(norms_out)
        self._H = None
        if host_grads is not None:
            if len(host_grads) != n:
                raise ValueError("host_grads must have one tensor per matrix")
            for h, g in zip(host_grads, grads):
                if h.shape != g.shape or h.dtype != g.dtype or not h.is_contiguous() or h.is_cuda:
                    raise ValueError("each host gradient must be a contiguous CPU tensor shaped and typed like its grad")
            self._keep = self._keep + (list(host_grads),)
            self._H = (ctypes.c_void_p * n)(*[t.data_ptr() for t in host_grads])
            self._groups = int(groups)

    def __call__(self, lr=0.02, beta=0.95, stream=None):
        if self._H is not None:
            _check(lib().dmuon_muon_step_host(self._n, self._P, self._H, self._G, self._gdtype, self._M, self._rows,
                                              self._cols, self._norms, float(lr), float(beta), self._coeffs,
                                              self._steps, self._restarts, self._nr, self._backend, self._eps,
                                              self._groups, _stream(stream)))
            return
        _check(lib().dmuon_muon_step(self._n, self._P, self._G, self._gdtype, self._M, self._rows, self._cols,
                                     self._norms, float(lr), float(beta), self._coeffs, self._steps, self._restarts,
                                     self._nr, self._backend, self._eps, _stream(stream)))


class AdamWStep:
    """AdamW over fixed tensors (the non-Muon parameters), prepared once; each call is one C call.

        adam = AdamWStep(params, grads, exp_avgs, exp_avg_sqs)
        adam(step=t, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01)
    """

    def __init__(self, params, grads, exp_avgs, exp_avg_sqs):
        n = len(params)
        if not (len(grads) == len(exp_avgs) == len(exp_avg_sqs) == n) or n == 0:
            raise ValueError("params, grads, exp_avgs and exp_avg_sqs must be non-empty lists of equal length")
        for p, g, m, v in zip(params, grads, exp_avgs, exp_avg_sqs):
            if not (p.numel() == g.numel() == m.numel() == v.numel()):
                raise ValueError("each param, grad and state must have the same number of elements")
            if not all(t.is_contiguous() for t in (p, g, m, v)):
                raise ValueError("tensors must be contiguous")
        self._keep = (list(params), list(grads), list(exp_avgs), list(exp_avg_sqs))
        self._n = n
        self._P = (ctypes.c_void_p * n)(*[_ptr(t) for t in params])
        self._G = (ctypes.c_void_p * n)(*[_ptr(t) for t in grads])
        self._M = (ctypes.c_void_p * n)(*[_ptr(t) for t in exp_avgs])
        self._V = (ctypes.c_void_p * n)(*[_ptr(t) for t in exp_avg_sqs])
        self._numel = (ctypes.c_int64 * n)(*[t.numel() for t in params])
        self._gdtype = _grad_dtype(grads)

    def __call__(self, step, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01, stream=None):
        _check(lib().dmuon_adamw_step(self._n, self._P, self._G, self._gdtype, self._M, self._V, self._numel,
                                      float(lr), float(betas[0]), float(betas[1]), float(eps), float(weight_decay),
                                      int(step), _stream(stream)))


def adamw_step(params, grads, exp_avgs, exp_avg_sqs, step, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01,
               stream=None):
    """One AdamW step over lists of CUDA tensors (fp32 params and states, fp32 or bf16 grads)."""
    AdamWStep(params, grads, exp_avgs, exp_avg_sqs)(step, lr, betas, eps, weight_decay, stream)


def momentum_normalize(grads, momenta, x_out, norms_out, beta=0.95, eps=1e-7, stream=None):
    """M <- beta M + G (grads may be None), norms_out[i] = ||M_i||, x_out[i] = fp16(M_i / (||M_i|| + eps)),
    oriented so rows <= cols."""
    n = len(momenta)
    gd = F32 if grads is None else _grad_dtype(grads)
    G = None if grads is None else (ctypes.c_void_p * n)(*[_ptr(t) for t in grads])
    M = (ctypes.c_void_p * n)(*[_ptr(t) for t in momenta])
    X = (ctypes.c_void_p * n)(*[_ptr(t) for t in x_out])
    rows = (ctypes.c_int64 * n)(*[t.shape[0] for t in momenta])
    cols = (ctypes.c_int64 * n)(*[t.shape[1] for t in momenta])
    _check(lib().dmuon_momentum_normalize(n, G, gd, M, rows, cols, X, _ptr(norms_out), float(beta), float(eps),
                                          _stream(stream)))


def momentum_normalize_noalloc(grad, momentum, x_out, norm_out, beta=0.95, eps=1e-7, stream=None):
    """One matrix of momentum_normalize with no device allocation (fixed library scratch); grad may be
    None. For callers whose device memory is owned by someone else."""
    gd = F32 if grad is None else _grad_dtype([grad])
    _check(lib().dmuon_momentum_normalize_noalloc(_ptr(grad), gd, _ptr(momentum), momentum.shape[0],
                                                  momentum.shape[1], _ptr(x_out), _ptr(norm_out), float(beta),
                                                  float(eps), _stream(stream)))


def gemm_f16(a, b, d, b_trans=True, e=None, alpha=1.0, beta=0.0, gamma=0.0, symmetric=False, stream=None):
    """D = fp16(alpha * A Bop + beta * E + gamma * I), Bop = B^T (b_trans) or B. fp16 CUDA tensors,
    rows contiguous (leading dimension = stride(0))."""
    M, K = a.shape
    N = b.shape[0] if b_trans else b.shape[1]
    _check(lib().dmuon_gemm_f16(M, N, K, _ptr(a), a.stride(0), _ptr(b), b.stride(0), 1 if b_trans else 0, _ptr(e),
                                e.stride(0) if e is not None else 0, _ptr(d), d.stride(0), float(alpha), float(beta),
                                float(gamma), 1 if symmetric else 0, _stream(stream)))
    return d


def check_status(stream=None):
    """Synchronise the stream and raise DmuonError if a kernel reported a timeout or a non-finite value."""
    _check(lib().dmuon_check_status(_stream(stream)))


def set_workspace_limit(nbytes):
    _check(lib().dmuon_set_workspace_limit(int(nbytes)))


def workspace_size(shapes, backend="gram"):
    n = len(shapes)
    rows = (ctypes.c_int64 * n)(*[s[0] for s in shapes])
    cols = (ctypes.c_int64 * n)(*[s[1] for s in shapes])
    out = ctypes.c_size_t(0)
    _check(lib().dmuon_workspace_size(n, rows, cols, _backend(backend), ctypes.byref(out)))
    return out.value


def set_graph_replay(on=True):
    """Graph replay of repeated calls (on by default): the second consecutive call with the same plan and
    arguments is captured as a CUDA graph and later such calls launch it; off launches every call directly."""
    _check(lib().dmuon_set_graph_replay(1 if on else 0))


def timing_enable(on=True):
    """Record CUDA events around every library launch (on the launching stream) until disabled."""
    _check(lib().dmuon_timing_enable(1 if on else 0))


def timing_read():
    """{class: (milliseconds, launches)} since the last read; waits for the recorded events."""
    ms = (ctypes.c_double * len(TIMING_CLASSES))()
    n = (ctypes.c_int64 * len(TIMING_CLASSES))()
    _check(lib().dmuon_timing_read(ms, n))
    return {c: (ms[i], n[i]) for i, c in enumerate(TIMING_CLASSES)}


def timing_read_launches(max_launches=4096):
    """[(class, milliseconds)] launch by launch, in launch order, since the last read (at most
    max_launches are returned); waits for the recorded events and clears the record."""
    ms = (ctypes.c_double * max_launches)()
    cls = (ctypes.c_int * max_launches)()
    n = ctypes.c_int()
    _check(lib().dmuon_timing_read_launches(max_launches, ms, cls, ctypes.byref(n)))
    return [(TIMING_CLASSES[cls[i]] if 0 <= cls[i] < len(TIMING_CLASSES) else str(cls[i]), ms[i])
            for i in range(min(n.value, max_launches))]


def selftest_bounded_wait(seconds=0.05, stream=None):
    """Launch one bounded wait that cannot complete (limit `seconds`): the next check_status() raises
    DmuonError with status ERR_TIMEOUT, exactly as when one of the library's waits runs out."""
    _check(lib().dmuon_selftest_bounded_wait(int(seconds * 1e9), _stream(stream)))


def selftest_range_check(stream=None):
    """Checked build only: launch one GEMM whose only tile lies outside its product; the next
    check_status() raises DmuonError with status ERR_RANGE. The regular build raises ERR_UNSUPPORTED."""
    _check(lib().dmuon_selftest_range_check(_stream(stream)))


def plan_info():
    """(executed MMA flops, tiles, GEMM launches) of one run of the current device's cached plan."""
    f, t, n = ctypes.c_double(), ctypes.c_int64(), ctypes.c_int()
    _check(lib().dmuon_plan_info(ctypes.byref(f), ctypes.byref(t), ctypes.byref(n)))
    return f.value, t.value, n.value


def assign_owners(shapes, nranks, layer_ids=None, cost="gram_flops"):
    """Dedicated ownership by LPT (host-only): returns (owner rank per matrix, summed cost per rank)."""
    n = len(shapes)
    rows = (ctypes.c_int64 * n)(*[s[0] for s in shapes])
    cols = (ctypes.c_int64 * n)(*[s[1] for s in shapes])
    layers = None if layer_ids is None else (ctypes.c_int * n)(*[int(x) for x in layer_ids])
    owners = (ctypes.c_int * n)()
    loads = (ctypes.c_double * nranks)()
    _check(lib().dmuon_assign_owners(n, rows, cols, layers, int(nranks), COST_MODELS[cost], owners, loads))
    return list(owners), list(loads)


def release_workspace():
    _check(lib().dmuon_release_workspace())


def gram_flops(m, n, steps=5, restarts=DEFAULT_RESTARTS, dense=False, s_symmetric=True):
    """Flops of Gram NS on one matrix (m <= n after orientation), every symmetric product counted at half:
    X X^T m^2 n; per step R^2 m^3, the Q update Z Q 2 m^3 unless right after a (re)start, the R update
    R <- (aI+Z) R (aI+Z) when the next step exists and is not a restart; restart Q X 2 m^2 n + X X^T m^2 n;
    output Q X 2 m^2 n.

    The R update is S = (aI+Z) R followed by R = S (aI+Z) (symmetric, m^3). With s_symmetric=True (the
    library's execution: S is also symmetric in exact arithmetic and computed as an upper triangle plus
    mirror) S costs m^3, and the default 5 steps with restart [2] give 6 m^2 n + 17 m^3. With
    s_symmetric=False S is counted as the full product it is written as (2 m^3), the algorithmic count of
    the method as stated: 6 m^2 n + 20 m^3. dense=True counts every symmetric product in full (8 m^2 n +
    28 m^3 with the defaults), the count a general GEMM would execute."""
    m, n = min(m, n), max(m, n)
    h = 2 if dense else 1  # symmetric products: half, or in full
    hs = h if s_symmetric else 2
    rs = {k for k in restarts if 0 < k < steps}
    f, fresh = h * m * m * n, True
    for k in range(steps):
        if k in rs:
            f += 2 * m * m * n + h * m * m * n
            fresh = True
        f += h * m ** 3 + (0 if fresh else 2 * m ** 3)
        fresh = False
        if k + 1 < steps and (k + 1) not in rs:
            f += (hs + h) * m ** 3
    return f + 2 * m * m * n


def auto_uses_direct(m, n):
    """The auto backend's per-matrix choice: direct when its flops are below Gram's (n < 4m/3)."""
    m, n = min(m, n), max(m, n)
    return 3 * n < 4 * m


def direct_flops(m, n, steps=5, dense=False):
    """Algorithmic flops of direct NS on one matrix, symmetric products at half: per step
    X X^T m^2 n, A^2 m^3, B X 2 m^2 n (dense=True: the symmetric ones in full, 4 m^2 n + 2 m^3)."""
    m, n = min(m, n), max(m, n)
    h = 2 if dense else 1
    return steps * ((h + 2) * m * m * n + h * m ** 3)


def __getattr__(name):
    """newton_schulz, NewtonSchulz, Muon and default_muon_filter load from .optim on first use (it imports
    torch; this module does not)."""
    if name in ("newton_schulz", "NewtonSchulz", "Muon", "default_muon_filter"):
        from . import optim
        return getattr(optim, name)
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")
