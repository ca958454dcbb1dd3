"""Benchmark: one owner-rank Muon step over the Muon-target matrices of a Llama-3-8B-shaped model.

A step is the whole path on every matrix: momentum accumulate (bf16 gradients, fp32 momentum), fp32
Frobenius normalisation, fp16 cast, five Newton-Schulz steps (Gram form with restart [2] by default,
POLAR_EXPRESS coefficients) and the fp32 weight update -- one dmuon_muon_step call.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--backend gram|direct] [--layers L]
    python bench.py --impl reference ...   # the CPU float64 oracle on a bounded sample

value = algorithmic Newton-Schulz TFLOP/s of the whole job (every symmetric product counted at half:
Gram as implemented 6 m^2 n + 17 m^3 per matrix -- R, Z and S = (aI+Z)R are symmetric, Q is a full
product --, direct 15 m^2 n + 5 m^3) over the device-timed region, inputs resident in HBM. Every input is larger than L2 (129 MB) except the small Gram matrices, so no flush is inserted.
e2e = the same metric through the public call a caller with host gradients makes
(dmuon_muon_step_host: the step's gradients copied in from pinned host memory inside the call, the copies
pipelined against the computation) and the per-matrix norms read back, inside the timed region.
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
UNIT = "TFLOP/s"
LR, BETA, EPS = 0.02, 0.95, 1e-7


def parse():
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
                         "adamw: AdamW over the Llama-3-8B non-Muon parameters; ns-configs: the single "
                         "256x1024 matrix and the closed-form 4096^2 and 2048x8192 dmuon_ns cases, both forms")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--e2e-groups", type=int, default=0,
                    help="pipeline groups of the host-gradient call (0: the library's choice, 1: no overlap)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline (profiling runs)")
    ap.add_argument("--torch-mm-context", action="store_true",
                    help="time the same step written with torch.mm (cuBLAS) instead; context only")
    return ap.parse_args()


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


def total_flops(shapes, backend, restarts=(2,), dense=False):
    import newton_schulz_momentum_gb300 as dm

    def one(r, c):
        direct = backend == "direct" or (backend == "auto" and dm.auto_uses_direct(r, c))
        return dm.direct_flops(r, c, dense=dense) if direct else dm.gram_flops(r, c, 5, restarts, dense=dense)
    return sum(one(r, c) for _, r, c in shapes)


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


def cpu_oracle_sample(shapes, backend, seconds, seed=7, small=False):
    """Time the float64 oracle (as it stands) on whole matrices of the workload's distinct oriented
    shapes, cycling until about `seconds` of CPU work. Returns (TFLOP/s, flops, seconds, sample text)."""
    import numpy as np

    import newton_schulz_momentum_gb300 as dm
    import workloads
    from oracle import ns64

    distinct = []
    for name, r, c in shapes:
        key = (min(r, c), max(r, c))
        if key not in [(min(a, b), max(a, b)) for _, a, b in distinct]:
            distinct.append((name, r, c))
    distinct.sort(key=lambda t: t[1] * t[2])
    flops, spent, done = 0, 0.0, []
    i = 0
    while spent < seconds or not done:
        name, r, c = distinct[i % len(distinct)]
        g = workloads.gaussian((r, c), 1e-3, seed + i)
        if not small:
            g = workloads.round_to_bf16(g)[0]
        w = workloads.gaussian((r, c), 0.02, seed + 100 + i)
        m0 = np.zeros((r, c), dtype=np.float32)
        coeffs = ns64.YOU if small else ns64.POLAR_EXPRESS
        t0 = time.perf_counter()
        ns64.muon_step(w, g, m0, LR, BETA, coeffs, (2,) if backend == "gram" else (), backend, EPS)
        spent += time.perf_counter() - t0
        flops += (dm.gram_flops if backend == "gram" else dm.direct_flops)(r, c)
        done.append(f"{name.split('.')[-1]} {r}x{c}")
        i += 1
        if i >= 3 * len(distinct) and not small:
            break
    return flops / spent / 1e12, flops, spent, "whole-matrix oracle Muon steps: " + ", ".join(done)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    """--impl reference: the CPU float64 oracle on the same workload, metric and unit."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    shapes, cfg = workload_config(args)
    per_step = max(args.cpu_seconds / 4.0, 1.0)
    for _ in range(args.warmup):
        cpu_oracle_sample(shapes[:7], args.backend, 0.0, small=args.workload == "small")
    tflops, flops, secs = [], 0, 0.0
    sample = ""
    for _ in range(args.steps):
        v, f, s, sample = cpu_oracle_sample(shapes[:7], args.backend, per_step, small=args.workload == "small")
        tflops.append(v)
        flops += f
        secs += s
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                         "sample": f"per step about {per_step:.0f} s of {sample}"},
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

    shapes, cfg = workload_config(args)
    flops_step = total_flops(shapes, args.backend, restart_list(args))
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

    muon = dm.MuonStep(W, G, M, coeffs=coeffs, restarts=restart_list(args), backend=args.backend, eps=EPS,
                       norms_out=norms)
    cuda_stream = stream.cuda_stream

    def step():
        muon(lr=LR, beta=BETA, stream=cuda_stream)

    def make_host_step(host_grads):
        host_muon = dm.MuonStep(W, G, M, coeffs=coeffs, restarts=restart_list(args), backend=args.backend, eps=EPS,
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
    value = whole_job_tflops(flops_step, world, ms_step)
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

    # ---- roofline of the dominant kernel (the tensor-core GEMM), from the live events
    hbm, tc_burst, tc_sust, src = peaks()
    gemm_ms, gemm_n = kernel_times["gemm_tc"]
    per_launch_flops = flops_step * args.steps / max(gemm_n, 1)
    achieved = per_launch_flops / (gemm_ms / max(gemm_n, 1) * 1e-3) / 1e12 if gemm_ms > 0 else None
    launches = sum(n for _, n in kernel_times.values())
    rw_ms = sum(kernel_times[k][0] for k in ("momentum_sumsq", "finalize_norms", "normalize_cast"))
    # momentum: G (2 B bf16 / 4 B fp32) + M read 4 + M write 4; normalise: M read 4 + X write 2 (no
    # separate normalise pass when the fused small-matrix kernel reads M itself)
    fused_small = kernel_times["normalize_cast"][1] == 0
    rw_bytes = (2 if gdtype == torch.bfloat16 else 4) + 4 + 4 + (0 if fused_small else 4 + 2)

    # dedicated ownership of this matrix set over 8 owner ranks (host-only LPT), timed and its balance
    layer_of = [int(name.split(".")[1]) if name.startswith("layers.") else 0 for name, _, _ in shapes]
    t0 = time.perf_counter()
    _, loads = dm.assign_owners([(r, c) for _, r, c in shapes], 8, layer_of, "gram_flops")
    owner_us = (time.perf_counter() - t0) * 1e6
    ownership = {"ranks": 8, "cost": "gram_flops", "max_over_mean_load": max(loads) / (sum(loads) / 8),
                 "host_us": owner_us}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v, f, s, sample = cpu_oracle_sample(shapes, args.backend, args.cpu_seconds, small=args.workload == "small")
        cpu = {"value": v, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": f"{sample} ({f / 1e12:.2f} TFLOP in {s:.1f} s, float64 NumPy)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic", "config": cfg,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": tc_sust, "unit": "TFLOP/s",
                         "frac": (achieved / tc_sust) if achieved else None,
                         "traffic": measured_traffic(cfg["workload"], args.backend),
                         "kernel": ("ns_small_kernel (whole fused iteration per matrix: tcgen05 fp16, fp32 "
                                    "accumulate; normalise/cast and weight update inside)") if fused_small
                         else "gemm_tc_kernel (tcgen05 fp16, fp32 accumulate)",
                         "peak_source": f"{src} bf16 sustained (fp16 dense rate equals bf16)"},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks.summary(),
            "breakdown_ms_per_step": {k: v[0] / args.steps for k, v in kernel_times.items()},
            "launches_per_step": {k: v[1] / args.steps for k, v in kernel_times.items()},
            "rowwise_hbm": {"bytes_per_step": sum(r * c for _, r, c in shapes) * rw_bytes,
                            "achieved_gbs": (sum(r * c for _, r, c in shapes) * rw_bytes * args.steps / (rw_ms * 1e-3) / 1e9)
                            if rw_ms > 0 else None, "peak_gbs": hbm,
                            "copy_gbs_this_box": live_copy_gbs},
            "ns_tflops_frac_of_peak": value / world / tc_sust,
            "step_ms": {"p50": statistics.median(per_step), "p90": per_step[min(len(per_step) - 1,
                                                                             int(0.9 * len(per_step)))],
                        "min": per_step[0], "max": per_step[-1]},
            "phases_ms_p50": phases,
            "dense_tflops": whole_job_tflops(total_flops(shapes, args.backend, restart_list(args), dense=True),
                                             world, ms_step),
            "executed": ({"tflop_per_step": exec_flops / 1e12, "tiles_per_step": exec_tiles,
                          "gemm_tflops": exec_flops * args.steps / (gemm_ms * 1e-3) / 1e12,
                          "frac_of_peak": exec_flops * args.steps / (gemm_ms * 1e-3) / 1e12 / tc_sust}
                         if exec_flops > 0 and gemm_ms > 0 else None),
            "owner_assignment": ownership,
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
    """The configurations beside the headline, timed one call at a time (CUDA events around each call on
    the current stream, median over --steps after --warmup): the single 256 x 1024 matrix (one Muon
    step, fp32 N(0, 1) gradient, YOU; latency-bound, reported in microseconds) and dmuon_ns on the
    closed-form 4096 x 4096 matrix (singular values log-uniform in [1e-6, 1]) and 2048 x 8192 matrix (205
    singular values 1, the rest 1e-4) with POLAR_EXPRESS, each in the Gram form (restart [2]) and the
    direct form; the 2048 x 8192 case also through dmuon_ns_tp split into 2 and 8 column shards. dmuon_ns
    works in place, so each call starts from a fresh copy of the input, made before
    its start event. Prints one JSON line."""
    import statistics

    import numpy as np
    import torch

    import newton_schulz_momentum_gb300 as dm
    import workloads

    dev = torch.device("cuda", 0)
    _, tc_burst, _, src = peaks()

    def timeit(fn, prep=None):
        marks = []
        for i in range(args.warmup + args.steps):
            if prep is not None:
                prep()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            if i >= args.warmup:
                marks.append((a, b))
        torch.cuda.synchronize(dev)
        ms = [a.elapsed_time(b) for a, b in marks]
        return statistics.median(ms), min(ms)

    out = []
    g = torch.from_numpy(workloads.gaussian((256, 1024), 1.0, 1)).to(dev)
    for backend in ("gram", "direct"):
        W, M = [torch.zeros((256, 1024), device=dev)], [torch.zeros((256, 1024), device=dev)]
        step = dm.MuonStep(W, [g], M, coeffs=dm.YOU, restarts=(2,), backend=backend)
        med, best = timeit(lambda: step(lr=LR, beta=BETA))
        dm.check_status()
        flops = dm.gram_flops(256, 1024) if backend == "gram" else dm.direct_flops(256, 1024)
        out.append({"config": "single 256x1024, Muon step, fp32 grad, YOU", "backend": backend,
                    "us_median": med * 1e3, "us_min": best * 1e3, "tflops": flops / (med * 1e-3) / 1e12,
                    "bound": "latency"})
    cases = (("4096x4096 closed form, sigma log-uniform in [1e-6, 1], POLAR_EXPRESS", 4096, 4096,
              workloads.log_uniform_spectrum(4096, 1e-6, 1.0, 2), 2),
             ("2048x8192 closed form, 205 sigma = 1, the rest 1e-4, POLAR_EXPRESS", 2048, 8192,
              workloads.top_fraction_spectrum(2048, 0.1, 1.0, 1e-4), 3))
    for name, m, n, sigma, seed in cases:
        x0 = torch.from_numpy(workloads.closed_form_matrix(m, n, sigma, seed)[0].astype(np.float32)).to(dev)
        x = torch.empty_like(x0)
        for backend in ("gram", "direct"):
            med, best = timeit(lambda: dm.ns(x, dm.POLAR_EXPRESS, (2,), backend), prep=lambda: x.copy_(x0))
            dm.check_status()
            flops = dm.gram_flops(m, n) if backend == "gram" else dm.direct_flops(m, n)
            tf = flops / (med * 1e-3) / 1e12
            out.append({"config": name, "backend": backend, "ms_median": med, "ms_min": best, "tflops": tf,
                        "bound": "tensor", "frac_of_burst_peak": tf / tc_burst})
        if m == 2048:
            # The column-split (tensor-parallel exact) Gram form emulated on this GPU: every Gram formation is
            # `shards` per-shard products written in fp32, then the fixed-order reduction.
            for shards in (2, 8):
                med, best = timeit(lambda: dm.ns_tp(x, shards, dm.POLAR_EXPRESS, (2,)), prep=lambda: x.copy_(x0))
                dm.check_status()
                tf = dm.gram_flops(m, n) / (med * 1e-3) / 1e12
                out.append({"config": name, "backend": f"gram, {shards} column shards (dmuon_ns_tp)",
                            "ms_median": med, "ms_min": best, "tflops": tf, "bound": "tensor",
                            "frac_of_burst_peak": tf / tc_burst})
    print(json.dumps({"impl": "native", "workload": "ns-configs", "steps": args.steps, "warmup": args.warmup,
                      "dtype": "f16", "data": "synthetic", "peak_tflops_burst": tc_burst,
                      "peak_source": f"{src} bf16 burst (fp16 dense rate equals bf16)", "results": out}),
          flush=True)


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
