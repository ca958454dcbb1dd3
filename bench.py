"""Benchmark: one owner-rank Muon step over the Muon-target matrices of a Llama-3-8B-shaped model.

A step is the whole path on every matrix: momentum accumulate (bf16 gradients, fp32 momentum), fp32
Frobenius normalisation, fp16 cast, five Newton-Schulz steps (Gram form with restart [2] by default,
POLAR_EXPRESS coefficients) and the fp32 weight update -- one dmuon_muon_step call.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--backend gram|direct] [--layers L] [--owned]
    python bench.py --impl reference ...   # the CPU float64 oracle, timed per matrix and extrapolated

value = algorithmic Newton-Schulz TFLOP/s of the whole job over the device-timed region, inputs resident
in HBM: Gram 6 m^2 n + 20 m^3 per matrix (the symmetric products X X^T, R^2 and R = S (aI+Z) counted at
half, S = (aI+Z) R as the full product the method writes), direct 15 m^2 n + 5 m^3. The library computes
S as a symmetric product too (it is one in exact arithmetic), so it executes 6 m^2 n + 17 m^3; the line
reports that count under "as_executed". Every input is larger than L2 (129 MB) except the small Gram
matrices, so no flush is inserted.
e2e = the same metric through the public call a caller with host gradients makes
(dmuon_muon_step_host: the step's gradients copied in from pinned host memory inside the call, the copies
pipelined against the computation) and the per-matrix norms read back, inside the timed region.
configs = the other configurations, each timed on its own with CUDA events and its own clock record:
the single 256 x 1024 matrix (both forms), the closed-form 4096 x 4096 and 2048 x 8192 matrices through
dmuon_ns (both forms), the 2560 small matrices in one grouped step, and the whole Llama-3-8B set in the
direct form.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Muon NS step ms & TFLOP/s (frac of fp16 tensor peak), 8B Llama matrix set"
SMALL_METRIC = "Muon NS step ms & TFLOP/s, 2560 small matrices (2048 x 128x512 + 512 x 512x128)"
UNIT = "TFLOP/s"
LR, BETA, EPS = 0.02, 0.95, 1e-7


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--backend", default="gram", choices=["gram", "direct", "auto"])
    ap.add_argument("--restarts", default="2", help="comma-separated restart indices for the Gram form ('' for none)")
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--workload", default="llama", choices=["llama", "small", "adamw", "ns-configs"],
                    help="llama: Llama-3-8B Muon-target set (the headline); small: 2048 x 128x512 + 512 x 512x128; "
                         "adamw: AdamW over the Llama-3-8B non-Muon parameters; ns-configs: only the other "
                         "configurations (the single 256x1024 matrix, the closed-form dmuon_ns cases, the small "
                         "set, the 8B set in the direct form)")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--e2e-groups", type=int, default=0,
                    help="pipeline groups of the host-gradient call (0: the library's choice, 1: no overlap)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline (profiling runs)")
    ap.add_argument("--config-steps", type=int, default=10,
                    help="timed calls per other configuration (0: skip them)")
    ap.add_argument("--owned", action="store_true",
                    help="dedicated ownership across the ranks: each rank updates only the matrices "
                         "dmuon_assign_owners gives it (LPT over Gram flops, same-layer spread), so the job "
                         "is one matrix set (strong scaling) instead of one per rank")
    ap.add_argument("--torch-mm-context", action="store_true",
                    help="time the same step written with torch.mm (cuBLAS) instead; context only")
    return ap.parse_args(argv)


def workload_config(args):
    import workloads
    if args.workload == "small":
        shapes = [(f"m{i}", r, c) for i, (r, c) in enumerate(workloads.small_set_shapes())]
        return shapes, {
            "workload": "small-set-2560", "matrices": len(shapes), "params": sum(r * c for _, r, c in shapes),
            "shapes": "2048 x 128x512 + 512 x 512x128", "grad_dtype": "fp32", "state_dtype": "fp32",
            "backend": args.backend, "coefficients": "YOU",
            "restarts": list(restart_list(args)) if args.backend != "direct" else [],
            "lr": LR, "beta": BETA, "eps": EPS, "l2": "inputs larger than L2, no flush",
        }
    shapes = workloads.llama3_8b_shapes(args.layers)
    return shapes, {
        "workload": f"llama3-8b-muon-set-{args.layers}L" if args.layers != 32 else "llama3-8b-muon-set",
        "matrices": len(shapes),
        "params": sum(r * c for _, r, c in shapes),
        "shapes": "per layer q/o 4096x4096, k/v 1024x4096, gate/up 14336x4096, down 4096x14336",
        "grad_dtype": "bf16", "state_dtype": "fp32", "backend": args.backend,
        "coefficients": "POLAR_EXPRESS", "restarts": list(restart_list(args)) if args.backend != "direct" else [],
        "lr": LR, "beta": BETA, "eps": EPS,
        "l2": "inputs larger than L2, no flush",
    }


def restart_list(args):
    return tuple(int(x) for x in args.restarts.split(",") if x.strip() != "")


def matrix_flops(r, c, backend, restarts=(2,), dense=False, as_executed=False):
    """Newton-Schulz flops of one matrix: the algorithmic count (Gram 6 m^2 n + 20 m^3 with the defaults,
    S = (aI+Z) R a full product), or with as_executed the library's (S symmetric: 6 m^2 n + 17 m^3);
    dense counts every symmetric product in full."""
    import newton_schulz_momentum_gb300 as dm
    direct = backend == "direct" or (backend == "auto" and dm.auto_uses_direct(r, c))
    if direct:
        return dm.direct_flops(r, c, dense=dense)
    return dm.gram_flops(r, c, 5, restarts, dense=dense, s_symmetric=as_executed)


def total_flops(shapes, backend, restarts=(2,), dense=False, as_executed=False):
    """matrix_flops summed over one step's matrices."""
    return sum(matrix_flops(r, c, backend, restarts, dense, as_executed) for _, r, c in shapes)


def owned_shapes(shapes, world, rank):
    """The matrices rank `rank` owns when `world` ranks split the set by dedicated ownership (LPT over
    Gram flops with the same-layer spread rule, computed identically on every rank)."""
    import newton_schulz_momentum_gb300 as dm
    layer_of = [int(name.split(".")[1]) if name.startswith("layers.") else 0 for name, _, _ in shapes]
    owners, _ = dm.assign_owners([(r, c) for _, r, c in shapes], world, layer_of, "gram_flops")
    return [s for s, o in zip(shapes, owners) if o == rank]


# The GEMM's DRAM traffic depends on the kernel and on the planner's tile order.
# Per workload: the committed ncu DRAM capture of its dominant kernel, and the sources that kernel's
# traffic depends on (the capture is used only while their digest matches).
TRAFFIC = {
    "llama3-8b-muon-set": ("gemm_tc_dram_traffic.json", ("gemm_tc.cu", "tc_ptx.h", "internal.h", "api.cu")),
    "small-set-2560": ("ns_small_dram_traffic.json", ("ns_small.cu", "tc_ptx.h", "internal.h", "api.cu")),
}


def source_digest(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "newton_schulz_momentum_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(workload, backend):
    """DRAM bytes per launch of the workload's dominant kernel from the committed ncu capture, or None
    when there is none for this workload or it was taken on an earlier version of the kernel source."""
    if workload not in TRAFFIC:
        return None
    fname, files = TRAFFIC[workload]
    try:
        with open(os.path.join(ROOT, "profiles", fname)) as fh:
            rec = json.load(fh)
    except Exception:
        return None
    if rec.get("kernel_source_sha256") != source_digest(files):
        return None
    return rec.get("per_launch_bytes", {}).get(f"{workload}/{backend}")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"], "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_info():
    """The host CPU's model name and the BLAS library NumPy uses (what the oracle's matrix products run on)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as fh:
                for ln in fh:
                    if ln.lower().startswith(("model name", "cpu model")):
                        model = ln.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    import numpy as np
    blas = None
    try:
        deps = np.show_config(mode="dicts")["Build Dependencies"]
        b = deps.get("blas", {})
        blas = " ".join(str(b.get(k)) for k in ("name", "version") if b.get(k)) or None
    except Exception:
        pass
    return {"cpu_model": model, "blas": blas, "numpy": np.__version__}


def distinct_oriented(shapes):
    """[(rows, cols, count)]: one stored shape per distinct oriented shape (min, max), with how many of the
    workload's matrices have it, smallest first."""
    seen = {}
    for _, r, c in shapes:
        key = (min(r, c), max(r, c))
        if key not in seen:
            seen[key] = [r, c, 0]
        seen[key][2] += 1
    return sorted((tuple(v) for v in seen.values()), key=lambda t: t[0] * t[1])


def oracle_matrix_seconds(r, c, backend, small, seed):
    """Wall time of one oracle Muon step (float64 NumPy, as it stands) on one whole r x c matrix of the
    workload's distribution."""
    import numpy as np

    import workloads
    from oracle import ns64
    g = workloads.gaussian((r, c), 1e-3, seed)
    if not small:
        g = workloads.round_to_bf16(g)[0]
    w = workloads.gaussian((r, c), 0.02, seed + 100)
    m0 = np.zeros((r, c), dtype=np.float32)
    coeffs = ns64.YOU if small else ns64.POLAR_EXPRESS
    t0 = time.perf_counter()
    ns64.muon_step(w, g, m0, LR, BETA, coeffs, (2,) if backend == "gram" else (), backend, EPS)
    return time.perf_counter() - t0


def cpu_oracle_sample(shapes, backend, seconds, seed=7, small=False):
    """Time the float64 oracle on whole matrices of the workload's distinct oriented shapes (smallest
    first, cycling) until about `seconds` of CPU work. Returns (TFLOP/s on the algorithmic count, flops,
    seconds, sample text)."""
    distinct = distinct_oriented(shapes)
    flops, spent, done = 0, 0.0, {}
    i = 0
    # Large shapes take seconds each: at most three passes over the distinct shapes. Small ones take
    # milliseconds: as many as fit in the time budget.
    while (spent < seconds and (i < 3 * len(distinct) or small)) or not done:
        r, c, _ = distinct[i % len(distinct)]
        spent += oracle_matrix_seconds(r, c, backend, small, seed + i)
        flops += matrix_flops(r, c, backend)
        done[f"{r}x{c}"] = done.get(f"{r}x{c}", 0) + 1
        i += 1
    return (flops / spent / 1e12, flops, spent,
            "whole-matrix oracle Muon steps: " + ", ".join(f"{k} x {v}" for k, v in done.items()))


def run_reference(args):
    """--impl reference: the CPU float64 oracle (as it stands) on the same workload, metric and unit. Each
    timed step is one whole-matrix oracle Muon step, taking the workload's distinct oriented shapes in
    turn; the full step's time is extrapolated as the sum over the distinct shapes of (matrices of that
    shape x the mean measured time per matrix), since the whole 224-matrix step would take about twenty
    minutes of CPU time. value = the full step's algorithmic flops / that extrapolated time."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    shapes, cfg = workload_config(args)
    small = args.workload == "small"
    distinct = distinct_oriented(shapes)
    for i in range(args.warmup):
        oracle_matrix_seconds(distinct[0][0], distinct[0][1], args.backend, small, 11 + i)
    per_shape = {}
    wall = []
    for i in range(args.steps):
        r, c, _ = distinct[i % len(distinct)]
        t = oracle_matrix_seconds(r, c, args.backend, small, 21 + i)
        per_shape.setdefault((r, c), []).append(t)
        wall.append(t)
    sampled_flops = sum(matrix_flops(r, c, args.backend) * len(ts) for (r, c), ts in per_shape.items())
    rate = sampled_flops / sum(wall)  # flop/s over the sample, for shapes the sample did not reach
    step_s = 0.0
    for r, c, count in distinct:
        ts = per_shape.get((r, c))
        step_s += count * (statistics.mean(ts) if ts else matrix_flops(r, c, args.backend) / rate)
    flops_step = total_flops(shapes, args.backend)
    value = flops_step / step_s / 1e12
    sample = (f"{args.steps} whole-matrix oracle Muon steps, one per timed step, cycling the distinct oriented "
              f"shapes ({', '.join(f'{r}x{c}: {len(per_shape.get((r, c), []))}' for r, c, _ in distinct)}); "
              f"float64 NumPy")
    line = {
        "impl": "reference", "metric": SMALL_METRIC if small else METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * step_s,
        "ms_per_step_kind": "extrapolated: sum over the distinct shapes of matrices x mean measured oracle time "
                            "per matrix",
        "sample_ms_per_step": 1e3 * statistics.mean(wall),
        "per_shape_s": {f"{r}x{c}": {"matrices": count, "mean_s": statistics.mean(per_shape[(r, c)])
                                      if (r, c) in per_shape else None} for r, c, count in distinct},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle", "sample": sample,
                         **cpu_info()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def max_over_ranks(ms, device):
    """Largest per-rank time (ms) across the process group; the job is as slow as its slowest rank."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def live_copy_rate(dev):
    """This box's copy bandwidth measured the way the peaks file was (b.copy_(a) over 1 Gi bf16 elements,
    read + write bytes, best of 10): the row-wise passes are compared against it as well."""
    import torch
    a = torch.empty(1 << 30, dtype=torch.bfloat16, device=dev)
    b = torch.empty_like(a)
    a.fill_(1.0)
    best = None
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(11):
        e0.record()
        b.copy_(a)
        e1.record()
        e1.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None else min(best, ms)
    del a, b
    torch.cuda.empty_cache()
    return 2 * 2 * (1 << 30) / (best * 1e-3) / 1e9


def whole_job_tflops(flops_per_rank_step, world, ms_per_step):
    """Weak scaling: every rank updates its own full matrix set, so the job does world x the work."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def run_e2e(args, G, norms, make_host_step, barrier, stream, world, flops_step):
    """Same metric through the public call a caller with host gradients makes (dmuon_muon_step_host: the
    gradients are copied in from pinned host memory inside the call, pipelined against the computation),
    with the per-matrix norms (the step's reported result) read back, all inside the timed region."""
    import torch

    # Page-locked staging buffers (cudaHostAlloc) filled by the CPU, as a host that produces or stages
    # gradients fills them. On these coherently attached hosts, pinned pages last written by a GPU copy
    # (device-to-host) read back over DMA at about a third of the rate of CPU-written ones.
    host_g = [torch.empty(g.shape, dtype=g.dtype, pin_memory=True) for g in G]
    for h, g in zip(host_g, G):
        h.copy_(g.cpu())
    host_norms = torch.empty(norms.numel(), dtype=torch.float32).pin_memory()
    h2d = sum(g.numel() * g.element_size() for g in host_g)
    d2h = host_norms.numel() * host_norms.element_size()
    host_step = make_host_step(host_g)

    def e2e_step():
        host_step()
        host_norms.copy_(norms, non_blocking=True)

    # Untimed passes first, as for the device-resident steps: at least --warmup of them, then more (up to 12
    # in all) until two consecutive passes agree within 10%. Reads out of freshly filled pinned buffers run
    # several times slower for the first second or two (measured: 293, 268, 103 ms for the same 14 GB of
    # copies); a training loop reuses its staging buffers every step, so the settled rate is the one to time.
    wa, wb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    prev = None
    passes = 0
    for i in range(12):
        passes = i + 1
        wa.record(stream)
        e2e_step()
        wb.record(stream)
        wb.synchronize()
        t = wa.elapsed_time(wb)
        if i + 1 >= max(args.warmup, 1) and prev is not None and abs(t - prev) <= 0.1 * prev:
            break
        prev = t
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    start.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    stop.record(stream)
    barrier()
    ms = max_over_ranks(start.elapsed_time(stop), norms.device)
    # This machine's host link, measured on the same buffers right after (plain copies of every gradient, no
    # computation): the end-to-end step cannot beat max(device step, this copy time), and the link rate
    # differs a lot between hosts.
    la, lb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        la.record(stream)
        for g, h in zip(G, host_g):
            g.copy_(h, non_blocking=True)
        lb.record(stream)
    lb.synchronize()
    link_ms = la.elapsed_time(lb)
    del host_g
    return {"value": whole_job_tflops(flops_step, world, ms / args.e2e_steps), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms / args.e2e_steps,
            "warmup_passes": passes, "h2d_link_gbs_this_box": h2d / (link_ms * 1e-3) / 1e9,
            "h2d_copy_ms_this_box": link_ms}


def time_calls(fn, stream, dev, steps, prep=None):
    """CUDA-event times (ms) of `steps` calls of fn on `stream`, each bracketed by its own events (prep, if
    given, is enqueued before the start event and not timed): median, p90 and min."""
    import torch
    marks = []
    for _ in range(steps):
        if prep is not None:
            prep()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        marks.append((a, b))
    torch.cuda.synchronize(dev)
    ms = sorted(a.elapsed_time(b) for a, b in marks)
    return {"ms_median": statistics.median(ms), "ms_p90": ms[min(len(ms) - 1, int(0.9 * len(ms)))],
            "ms_min": ms[0], "calls": len(ms)}


def closed_form_on_device(m, n, sigma, seed, dev):
    """X = U diag(sigma) V^T as fp32 on the device, U (m x k) and V (n x k) orthonormal from the QR of seeded
    float64 Gaussians, k = min(m, n): the distribution of the closed-form parity cases, drawn on the GPU
    because NumPy's QR takes tens of seconds at these sizes (input generation only)."""
    import torch
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    k = min(m, n)

    def orth(rows):
        q, r = torch.linalg.qr(torch.randn((rows, k), generator=gen, device=dev, dtype=torch.float64))
        return q * torch.sign(torch.diagonal(r))
    u, v = orth(m), orth(n)
    s = torch.as_tensor(sigma, dtype=torch.float64, device=dev)
    return ((u * s) @ v.T).float().contiguous()


def run_configs(args, dev, local, big=None):
    """The configurations beside the headline, one at a time, each with a clock record: CUDA events around
    every call on the current stream, --config-steps timed calls after max(--warmup, 3) untimed ones.
      * Llama-3-8B set in the direct form (big = (shapes, W, G, M) of the headline, same buffers);
      * the 2560 small matrices (2048 x 128x512 + 512 x 512x128, fp32 N(0, 1e-3^2) gradients, YOU, Gram
        restart [2]) in one grouped step; HBM-bound: 20 B per element at least (G, M in; M out; W in and
        out), 24 B moved (the momentum pass, then the fused kernel reads M once more);
      * the single 256 x 1024 Muon step (fp32 N(0, 1) gradient, YOU), both forms; latency-bound;
      * dmuon_ns on the closed-form 4096 x 4096 matrix (singular values log-uniform in [1e-6, 1]) and
        2048 x 8192 matrix (205 singular values 1, the rest 1e-4), POLAR_EXPRESS, both forms; each call
        starts from a fresh copy of the input made before its start event.
    Flop rates use the algorithmic counts (Gram 6 m^2 n + 20 m^3 with restart [2], direct 15 m^2 n + 5 m^3)."""
    import torch

    import newton_schulz_momentum_gb300 as dm
    import workloads

    hbm, tc_burst, tc_sust, src = peaks()
    stream = torch.cuda.current_stream(dev)
    cs = stream.cuda_stream
    n = args.config_steps
    warm = max(args.warmup, 3)
    out = {"timing": f"CUDA events per call, median of {n} after {warm} untimed calls; peaks {src}"}

    def run(fn, prep=None, timing=False):
        """Warm-up calls, the timed calls (no per-launch events: an event recorded between two launches
        would stop the next one from starting while the previous drains), then, with timing, two more
        calls with per-launch events for the kernel split."""
        for _ in range(warm):
            if prep is not None:
                prep()
            fn()
        dm.check_status(stream)
        with ClockSampler(local) as clk:
            t = time_calls(fn, stream, dev, n, prep)
        kt = None
        if timing:
            dm.timing_enable(True)
            for _ in range(2):
                if prep is not None:
                    prep()
                fn()
            kt = {k: (ms / 2, c / 2) for k, (ms, c) in dm.timing_read().items()}
            dm.timing_enable(False)
        dm.check_status(stream)
        t["clocks"] = clk.summary()
        return t, kt

    if big is not None:
        shapes, W, G, M = big
        step = dm.MuonStep(W, G, M, coeffs=dm.POLAR_EXPRESS, restarts=(), backend="direct", eps=EPS)
        t, kt = run(lambda: step(lr=LR, beta=BETA, stream=cs), timing=True)
        flops = total_flops(shapes, "direct")
        gms, gn = kt["gemm_tc"]
        t.update({"config": "whole Llama-3-8B Muon-target set (224 matrices), bf16 grads, direct form, POLAR_EXPRESS",
                  "tflops": flops / (t["ms_median"] * 1e-3) / 1e12, "tflop_per_step": flops / 1e12,
                  "frac_of_sustained_peak": flops / (t["ms_median"] * 1e-3) / 1e12 / tc_sust,
                  "gemm_tc_ms_per_step": gms, "gemm_tc_launches_per_step": gn,
                  "gemm_tc_tflops": flops / (gms * 1e-3) / 1e12 if gms > 0 else None,
                  "kernel_split": "per-launch events on two further calls"})
        out["llama3_8b_direct"] = t
        del step

    # ---- the small-matrix set, one grouped step
    gen = torch.Generator(device=dev)
    gen.manual_seed(4)
    sshapes = workloads.small_set_shapes()
    W = [torch.randn(s, generator=gen, device=dev) * 0.02 for s in sshapes]
    G = [torch.randn(s, generator=gen, device=dev) * 1e-3 for s in sshapes]
    M = [torch.zeros(s, device=dev) for s in sshapes]
    step = dm.MuonStep(W, G, M, coeffs=dm.YOU, restarts=(2,), backend="gram", eps=EPS)
    t, kt = run(lambda: step(lr=LR, beta=BETA, stream=cs), timing=True)
    elems = sum(r * c for r, c in sshapes)
    flops = sum(matrix_flops(r, c, "gram") for r, c in sshapes)
    sec = t["ms_median"] * 1e-3
    t.update({"config": "2048 x 128x512 + 512 x 512x128 fp32 grads N(0, 1e-3^2), YOU, Gram restart [2], one grouped step",
              "elements": elems, "tflops": flops / sec / 1e12,
              "bytes_moved_per_step": 24 * elems, "gbs_moved": 24 * elems / sec / 1e9,
              "bytes_algorithmic_per_step": 20 * elems, "gbs_algorithmic": 20 * elems / sec / 1e9,
              "frac_of_hbm_algorithmic": 20 * elems / sec / 1e9 / hbm,
              "roofline_ms": max(20 * elems / (hbm * 1e9), flops / (tc_sust * 1e12)) * 1e3,
              "kernel_ms_per_step": {k: v[0] for k, v in kt.items() if v[1]},
              "launches_per_step": {k: v[1] for k, v in kt.items() if v[1]}})
    out["small_set_2560"] = t
    del step, W, G, M

    # ---- one 256 x 1024 matrix, the whole Muon step, both forms
    g = torch.from_numpy(workloads.gaussian((256, 1024), 1.0, 1)).to(dev)
    for backend in ("gram", "direct"):
        W1 = [torch.from_numpy(workloads.gaussian((256, 1024), 0.02, 2)).to(dev)]
        M1 = [torch.zeros((256, 1024), device=dev)]
        step = dm.MuonStep(W1, [g], M1, coeffs=dm.YOU, restarts=(2,), backend=backend, eps=EPS)
        t, kt = run(lambda: step(lr=LR, beta=BETA, stream=cs), timing=True)
        flops = matrix_flops(256, 1024, backend)
        t.update({"config": "single 256x1024 Muon step, fp32 N(0, 1) gradient, YOU", "bound": "latency",
                  "us_median": t["ms_median"] * 1e3, "tflops": flops / (t["ms_median"] * 1e-3) / 1e12,
                  "launches_per_step": {k: v[1] for k, v in kt.items() if v[1]}})
        out[f"single_256x1024_{backend}"] = t
        del step

    # ---- closed-form matrices through dmuon_ns
    cases = (("closed_form_4096x4096", "4096x4096, sigma log-uniform in [1e-6, 1], POLAR_EXPRESS", 4096, 4096,
              workloads.log_uniform_spectrum(4096, 1e-6, 1.0, 2), 2),
             ("closed_form_2048x8192", "2048x8192, 205 sigma = 1, the rest 1e-4, POLAR_EXPRESS", 2048, 8192,
              workloads.top_fraction_spectrum(2048, 0.1, 1.0, 1e-4), 3))
    for key, name, m, nn, sigma, seed in cases:
        x0 = closed_form_on_device(m, nn, sigma, seed, dev)
        x = torch.empty_like(x0)
        for backend in ("gram", "direct"):
            t, kt = run(lambda: dm.ns(x, dm.POLAR_EXPRESS, (2,), backend, EPS, stream=cs),
                        prep=lambda: x.copy_(x0), timing=True)
            flops = matrix_flops(m, nn, backend)
            tf = flops / (t["ms_median"] * 1e-3) / 1e12
            t.update({"config": f"dmuon_ns {name}", "bound": "tensor", "tflops": tf,
                      "frac_of_burst_peak": tf / tc_burst,
                      "launches_per_call": {k: v[1] for k, v in kt.items() if v[1]}})
            out[f"{key}_{backend}"] = t
        del x0, x
    torch.cuda.empty_cache()
    return out


def run_native(args):
    import torch
    import torch.distributed as dist

    import newton_schulz_momentum_gb300 as dm
    from newton_schulz_momentum_gb300 import build as dmbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    dmbuild.build()
    dm.lib()

    all_shapes, cfg = workload_config(args)
    shapes = owned_shapes(all_shapes, world, rank) if args.owned else all_shapes
    if args.owned:
        cfg = dict(cfg, ownership=f"dedicated: {world} ranks, LPT over Gram flops (dmuon_assign_owners)")
    restarts = restart_list(args)
    flops_step = total_flops(shapes, args.backend, restarts)  # this rank's matrices
    flops_job = total_flops(all_shapes, args.backend, restarts) if args.owned else world * flops_step
    flops_exec = total_flops(shapes, args.backend, restarts, as_executed=True)
    dev = torch.device("cuda", local)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    W, G, M = [], [], []
    gdtype = torch.float32 if args.workload == "small" else torch.bfloat16
    coeffs = dm.YOU if args.workload == "small" else dm.POLAR_EXPRESS
    for _, r, c in shapes:
        W.append(torch.randn((r, c), generator=gen, device=dev) * 0.02)
        G.append((torch.randn((r, c), generator=gen, device=dev) * 1e-3).to(gdtype))
        M.append(torch.zeros((r, c), dtype=torch.float32, device=dev))
    norms = torch.empty(len(shapes), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    muon = dm.MuonStep(W, G, M, coeffs=coeffs, restarts=restarts, backend=args.backend, eps=EPS, norms_out=norms)
    cuda_stream = stream.cuda_stream

    def step():
        muon(lr=LR, beta=BETA, stream=cuda_stream)

    def make_host_step(host_grads):
        host_muon = dm.MuonStep(W, G, M, coeffs=coeffs, restarts=restarts, backend=args.backend, eps=EPS,
                                norms_out=norms, host_grads=host_grads, groups=args.e2e_groups)
        return lambda: host_muon(lr=LR, beta=BETA, stream=cuda_stream)

    for _ in range(args.warmup):
        step()
    dm.check_status(stream)
    live_copy_gbs = live_copy_rate(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ---- device-resident timed region (an event before every step for the per-step spread)
    dm.timing_enable(True)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    barrier()
    with ClockSampler(local) as clocks:
        start.record(stream)
        for i in range(args.steps):
            marks[i].record(stream)
            step()
        marks[args.steps].record(stream)
        stop.record(stream)
        barrier()
    launch_list = dm.timing_read_launches(64 * args.steps + 64)
    dm.timing_enable(False)
    dm.check_status(stream)
    exec_flops, exec_tiles, _ = dm.plan_info()
    ms_step = max_over_ranks(start.elapsed_time(stop), dev) / args.steps
    value = flops_job / (ms_step * 1e-3) / 1e12
    per_step = sorted(marks[i].elapsed_time(marks[i + 1]) for i in range(args.steps))
    kernel_times = {c: (sum(ms for k, ms in launch_list if k == c), sum(1 for k, _ in launch_list if k == c))
                    for c in dm.TIMING_CLASSES}
    # per launch position within a step (the phases, in order): median over the timed steps
    phases = None
    if launch_list and len(launch_list) % args.steps == 0:
        lps = len(launch_list) // args.steps
        phases = [[launch_list[j][0], statistics.median(launch_list[i * lps + j][1] for i in range(args.steps))]
                  for j in range(lps)]

    # ---- end to end through the public call: pinned host gradients in, norms out
    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(args, G, norms, make_host_step, barrier, stream, world, flops_step)
        if args.owned:
            e2e["value"] = flops_job / (e2e["ms_per_step"] * 1e-3) / 1e12

    # ---- roofline of the dominant kernel (the tensor-core GEMM), from the live events
    hbm, tc_burst, tc_sust, src = peaks()
    gemm_ms, gemm_n = kernel_times["gemm_tc"]
    per_launch_flops = flops_step * args.steps / max(gemm_n, 1)
    achieved = per_launch_flops / (gemm_ms / max(gemm_n, 1) * 1e-3) / 1e12 if gemm_ms > 0 else None
    launches = sum(n for _, n in kernel_times.values())
    rw_ms = sum(kernel_times[k][0] for k in ("momentum_sumsq", "finalize_norms", "normalize_cast"))
    # momentum: G (2 B bf16 / 4 B fp32) + M read 4 + M write 4; normalise: M read 4 + X write 2 (no
    # separate normalise pass when the fused small-matrix kernel reads M itself). The algorithmic minimum
    # reads G and M once and writes M and X once: 12 B (bf16 G) or 14 B (fp32 G) per element.
    fused_small = kernel_times["normalize_cast"][1] == 0
    gsize = 2 if gdtype == torch.bfloat16 else 4
    rw_bytes = gsize + 4 + 4 + (0 if fused_small else 4 + 2)
    # With the fused small-matrix kernel the row-wise pass is the momentum alone, already at its minimum
    # (the fused kernel reads M again and builds X on chip: its bytes are that kernel's).
    rw_alg = rw_bytes if fused_small else gsize + 4 + 4 + 2
    elems = sum(r * c for _, r, c in shapes)
    if fused_small:
        # The fused kernel is bound by HBM (and latency), not the tensor pipe: its algorithmic bytes are
        # M read once (4 B) and W read and written once (8 B) per element.
        fused_bytes = 12 * elems
        fused_gbs = fused_bytes / (gemm_ms / max(gemm_n, 1) * 1e-3) / 1e9 if gemm_ms > 0 else None
        roofline = {"bound": "hbm", "achieved": fused_gbs, "peak": hbm, "unit": "GB/s",
                    "frac": (fused_gbs / hbm) if fused_gbs else None,
                    "traffic": measured_traffic(cfg["workload"], args.backend),
                    "algorithmic_bytes_per_launch": fused_bytes,
                    "kernel": ("ns_small_kernel (whole fused iteration per matrix: tcgen05 fp16, fp32 accumulate; "
                               "normalise/cast and weight update inside)"),
                    "peak_source": f"{src} HBM copy rate",
                    "tensor_view": {"achieved_tflops": achieved, "frac_of_sustained": (achieved / tc_sust)
                                    if achieved else None}}
    else:
        roofline = {"bound": "tensor", "achieved": achieved, "peak": tc_sust, "unit": "TFLOP/s",
                    "frac": (achieved / tc_sust) if achieved else None,
                    "traffic": measured_traffic(cfg["workload"], args.backend),
                    "kernel": "gemm_tc_kernel (tcgen05 fp16, fp32 accumulate)",
                    "peak_source": f"{src} bf16 sustained (fp16 dense rate equals bf16)"}

    # dedicated ownership of this matrix set over 8 owner ranks (host-only LPT), timed and its balance
    layer_of = [int(name.split(".")[1]) if name.startswith("layers.") else 0 for name, _, _ in all_shapes]
    t0 = time.perf_counter()
    _, loads = dm.assign_owners([(r, c) for _, r, c in all_shapes], 8, layer_of, "gram_flops")
    owner_us = (time.perf_counter() - t0) * 1e6
    ownership = {"ranks": 8, "cost": "gram_flops", "max_over_mean_load": max(loads) / (sum(loads) / 8),
                 "host_us": owner_us}

    # ---- the other configurations (one GPU only), then the CPU oracle baseline
    configs = None
    if world == 1 and args.config_steps > 0:
        configs = run_configs(args, dev, local, (shapes, W, G, M) if args.workload == "llama" else None)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v, f, s, sample = cpu_oracle_sample(shapes, args.backend, args.cpu_seconds, small=args.workload == "small")
        cpu = {"value": v, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": f"{sample} ({f / 1e12:.2f} TFLOP in {s:.1f} s, float64 NumPy)", **cpu_info()}

    if rank == 0:
        line = {
            "metric": METRIC if args.workload == "llama" else SMALL_METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True,
            "scaling": "strong" if args.owned else "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic", "config": cfg,
            "flop_count": ("algorithmic: Gram 6 m^2 n + 20 m^3 per matrix (symmetric products at half, "
                           "S = (aI+Z) R in full), direct 15 m^2 n + 5 m^3"),
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks.summary(),
            "as_executed": {"count": "Gram 6 m^2 n + 17 m^3 (S symmetric, as the library computes it)",
                            "tflop_per_step": flops_exec / 1e12,
                            "tflops": flops_exec * (flops_job / flops_step) / (ms_step * 1e-3) / 1e12,
                            "gemm_tflops": flops_exec * args.steps / (gemm_ms * 1e-3) / 1e12 if gemm_ms > 0 else None,
                            "gemm_frac_of_sustained_peak": flops_exec * args.steps / (gemm_ms * 1e-3) / 1e12 / tc_sust
                            if gemm_ms > 0 else None},
            "breakdown_ms_per_step": {k: v[0] / args.steps for k, v in kernel_times.items()},
            "launches_per_step": {k: v[1] / args.steps for k, v in kernel_times.items()},
            "rowwise_hbm": {"bytes_per_step": elems * rw_bytes,
                            "achieved_gbs": elems * rw_bytes * args.steps / (rw_ms * 1e-3) / 1e9 if rw_ms > 0 else None,
                            "algorithmic_bytes_per_step": elems * rw_alg,
                            "algorithmic_gbs": elems * rw_alg * args.steps / (rw_ms * 1e-3) / 1e9 if rw_ms > 0 else None,
                            "peak_gbs": hbm, "copy_gbs_this_box": live_copy_gbs},
            "ns_tflops_frac_of_peak": value / world / tc_sust,
            "step_ms": {"p50": statistics.median(per_step), "p90": per_step[min(len(per_step) - 1,
                                                                             int(0.9 * len(per_step)))],
                        "min": per_step[0], "max": per_step[-1]},
            "phases_ms_p50": phases,
            "dense_tflops": (total_flops(shapes, args.backend, restarts, dense=True) * (flops_job / flops_step)
                             / (ms_step * 1e-3) / 1e12),
            "executed": ({"tflop_per_step": exec_flops / 1e12, "tiles_per_step": exec_tiles,
                          "gemm_tflops": exec_flops * args.steps / (gemm_ms * 1e-3) / 1e12,
                          "frac_of_peak": exec_flops * args.steps / (gemm_ms * 1e-3) / 1e12 / tc_sust}
                         if exec_flops > 0 and gemm_ms > 0 else None),
            "owner_assignment": ownership,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_adamw(args):
    """AdamW over the non-Muon parameters of a Llama-3-8B-shaped model (1.05 G elements, bf16 grads):
    HBM-bound, reported as GB/s of the bytes each element needs (p, g, m, v in; p, m, v out: 26 B)."""
    import torch

    import newton_schulz_momentum_gb300 as dm
    import workloads
    from newton_schulz_momentum_gb300 import build as dmbuild

    dmbuild.build()
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(77)
    numels = [n for _, n in workloads.llama3_8b_non_muon_numels()]
    P = [torch.randn(n, generator=gen, device=dev) * 0.02 for n in numels]
    G = [(torch.randn(n, generator=gen, device=dev) * 1e-3).to(torch.bfloat16) for n in numels]
    M = [torch.zeros(n, device=dev) for n in numels]
    V = [torch.zeros(n, device=dev) for n in numels]
    adam = dm.AdamWStep(P, G, M, V)
    stream = torch.cuda.current_stream(dev)
    for t in range(1, args.warmup + 1):
        adam(t, stream=stream)
    dm.check_status(stream)
    dm.timing_enable(True)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    with ClockSampler(0) as clocks:
        start.record(stream)
        for t in range(args.warmup + 1, args.warmup + args.steps + 1):
            adam(t, stream=stream)
        stop.record(stream)
        torch.cuda.synchronize(dev)
    kt = dm.timing_read()
    dm.timing_enable(False)
    dm.check_status(stream)
    ms = start.elapsed_time(stop) / args.steps
    nbytes = sum(numels) * 26
    hbm, _, _, src = peaks()
    kms, kn = kt["adamw"]
    achieved = nbytes / (kms / kn * 1e-3) / 1e9 if kn else None  # one launch per step: bytes / launch time
    line = {
        "metric": "AdamW step GB/s, Llama-3-8B non-Muon parameters", "value": nbytes / (ms * 1e-3) / 1e9,
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "llama3-8b-non-muon-adamw", "tensors": len(numels), "elements": sum(numels),
                   "grad_dtype": "bf16", "bytes_per_element": 26, "l2": "inputs larger than L2, no flush"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm if achieved else None, "traffic": None, "kernel": "adamw_kernel",
                     "peak_source": src},
        "gpu_launches": kn, "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


def run_torch_mm_context(args):
    """Context only, not the product path: the same step (momentum, norm, fp16 Gram NS with restart [2],
    W update) written with torch.mm (cuBLAS fp16 GEMMs, fp32 accumulation) one matrix at a time, timed
    like the native arm. Prints one JSON line with "impl": "torch-mm-context"."""
    import torch

    import newton_schulz_momentum_gb300 as dm

    shapes, cfg = workload_config(args)
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    W = [torch.randn((r, c), generator=gen, device=dev) * 0.02 for _, r, c in shapes]
    G = [(torch.randn((r, c), generator=gen, device=dev) * 1e-3).to(torch.bfloat16) for _, r, c in shapes]
    M = [torch.zeros((r, c), device=dev) for _, r, c in shapes]
    coeffs = dm.POLAR_EXPRESS
    restarts = set(restart_list(args))

    def ns(x):
        eye = torch.eye(x.shape[0], device=dev, dtype=torch.float16)
        r = x @ x.T
        q = eye.clone()
        for k, (a, b, c) in enumerate(coeffs):
            if k in restarts and k > 0:
                x = q @ x
                r = x @ x.T
                q = eye.clone()
            z = b * r + c * (r @ r)
            q = z @ q + a * q
            if k + 1 < len(coeffs) and (k + 1) not in restarts:
                w = z + a * eye
                r = (w @ r) @ w
        return q @ x

    def step():
        for w, g, m in zip(W, G, M):
            m.mul_(BETA).add_(g.float())
            x = (m / (m.norm() + EPS)).half()
            t = x.shape[0] > x.shape[1]
            o = ns(x.T if t else x)
            w.add_((o.T if t else o).float(), alpha=-LR)

    for _ in range(args.warmup):
        step()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    start.record()
    for _ in range(args.steps):
        step()
    stop.record()
    torch.cuda.synchronize(dev)
    ms = start.elapsed_time(stop) / args.steps
    flops = total_flops(shapes, "gram", restart_list(args))
    print(json.dumps({"impl": "torch-mm-context", "metric": METRIC, "value": flops / (ms * 1e-3) / 1e12,
                      "unit": UNIT, "ms_per_step": ms, "steps": args.steps, "warmup": args.warmup,
                      "config": cfg, "note": "cuBLAS fp16 via torch.mm, one matrix at a time; same algorithm "
                      "and flop count as the native arm; context only"}), flush=True)


def run_ns_configs(args):
    """--workload ns-configs: only the other configurations (run_configs), without the headline step;
    prints one JSON line."""
    import torch

    from newton_schulz_momentum_gb300 import build as dmbuild
    dmbuild.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    print(json.dumps({"impl": "native", "workload": "ns-configs", "dtype": "f16", "data": "synthetic",
                      "configs": run_configs(args, dev, 0)}), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.torch_mm_context:
        run_torch_mm_context(args)
    elif args.workload == "adamw":
        run_adamw(args)
    elif args.workload == "ns-configs":
        run_ns_configs(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
