#!/usr/bin/env python
"""Benchmark of the 1-bit LAMB hot path on GB300.

One step = one compression-stage step of the whole hot path (fused worker +
server compression over all W workers, per-tensor factor, frozen-variance
update) over the workload's full parameter table, through the C ABI.
Gradients are regenerated on the device before every step, outside the
CUDA-event-timed region (so every step sees new gradients and the L2 is
flushed between steps: each step moves ~80 GB, far above the 129 MB L2).

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workload  # noqa: E402  (seeded synthetic inputs; no optimizer arithmetic)

METRIC = "compression-stage param elements/s per step and achieved HBM GB/s vs GB300 peak"
UNIT = "params/s"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="large",
                   choices=("tiny", "base", "large", "large_w32", "gpt2xl"))
    p.add_argument("--variant", choices=("lamb", "adam"), default="lamb",
                   help="1-bit LAMB (default) or the 1-bit Adam variant")
    p.add_argument("--errors", choices=("f32", "bf16"), default="f32",
                   help="storage of the worker and server error buffers")
    p.add_argument("--chunk", type=int, default=0,
                   help="override the workload's chunk size C (the named workloads fix it)")
    p.add_argument("--workers", type=int, default=0,
                   help="override the workload's worker count W (the named workloads fix it)")
    p.add_argument("--first-tensor", type=int, default=0,
                   help="drop the tensors before this index of the table (profiling)")
    p.add_argument("--max-params", type=int, default=0,
                   help="keep only the leading tensors up to this many parameters (profiling)")
    p.add_argument("--warmup-stage-steps", type=int, default=-1,
                   help="LAMB warmup steps before the freeze (default: the workload's)")
    p.add_argument("--e2e-steps", type=int, default=6)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    return p.parse_args()


def get_workload(args):
    wl = workload.workloads()[args.workload]
    if args.chunk:
        wl.chunk = args.chunk
        wl.name = f"{wl.name}[C={args.chunk}]"
    if args.workers:
        wl.W = args.workers
        wl.name = f"{wl.name}[W={args.workers}]"
    if args.first_tensor:
        wl.tensors = wl.tensors[args.first_tensor:]
        wl.name = f"{wl.name}[{args.first_tensor}:]"
    if args.max_params:
        keep, n = [], 0
        for name, shape in wl.tensors:
            size = int(np.prod(shape))
            if keep and n + size > args.max_params:
                break
            keep.append((name, shape))
            n += size
        wl.tensors = keep
        wl.name = f"{wl.name}[:{n}]"
    return wl


def grad_bytes(wl):
    return {"f32": 4, "bf16": 2, "philox": 0}[wl.grad]


def fused_kernel_bytes(wl, variant="lamb", errors="f32"):
    """Algorithmic HBM bytes of one steady-state launch of the fused
    compression kernel: per parameter W*(g + 4 e_w read + 4 e_w written + 1/8
    signs) + the previous step's server signs (1/8, the old momentum) + reads
    of 4 e_s + 4 v + 4 v_fresh and writes of 4 e_s + 4 v_fresh + 1/8 server
    signs; plus 4 bytes per scale (W worker scales and the server scale
    written, the previous server scale read)."""
    W = wl.W
    # 1-bit Adam reads and writes no second moments in this kernel; bfloat16
    # error storage moves 2 + 2 instead of 4 + 4 bytes per error element
    eb = 4.0 if errors == "bf16" else 8.0
    per = W * (grad_bytes(wl) + eb + 0.125) + (eb + 0.25 + (0.0 if variant == "adam" else 12.0))
    return wl.N * per + 4.0 * wl.K * (W + 2)


def update_kernel_bytes(wl):
    """Update kernel: server signs (1/8), v (4), x read and written (8)."""
    return wl.N * 12.125 + 4.0 * wl.K


def warmup_kernel_bytes(wl, variant="lamb"):
    """Warmup moments kernel: per parameter the W gradients, m and v read
    and written, and (1-bit LAMB, for the trust ratio's norms) x read."""
    return wl.N * (wl.W * grad_bytes(wl) + (16.0 if variant == "adam" else 20.0))


def warmup_stage_line(wl, variant, N, peak, warm_ms, kern_ms, layer_ms, upd_ms):
    """The warmup stage's per-step times (the first step, which builds
    nothing different but starts cold, is left out when there are more) and
    its two streaming kernels against the same peak as the compression
    stage (the warmup update moves m, v and x read, x written: 16 B)."""
    def avg(v):
        return statistics.mean(v[1:] or v)
    mk, uk = avg(kern_ms), avg(upd_ms)
    mb, ub = warmup_kernel_bytes(wl, variant), 16.0 * wl.N
    return {"ms_per_step": avg(warm_ms), "moments_kernel_ms": mk, "per_tensor_ms": avg(layer_ms),
            "update_ms": uk, "params_per_s": N / (avg(warm_ms) / 1e3),
            # in-kernel gradients: the moments kernel draws W values per element
            # and is bound by that arithmetic, not by HBM
            "moments_bound": "alu" if wl.grad == "philox" else "hbm",
            "moments_gbs": mb / (mk / 1e3) / 1e9, "moments_frac_of_peak": mb / (mk / 1e3) / 1e9 / peak,
            "update_gbs": ub / (uk / 1e3) / 1e9, "update_frac_of_peak": ub / (uk / 1e3) / 1e9 / peak,
            "steps": len(warm_ms)}


def step_bytes(wl, variant="lamb", errors="f32"):
    return fused_kernel_bytes(wl, variant, errors) + update_kernel_bytes(wl)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def code_tokens(text):
    """C/C++ source with its comments removed and every run of whitespace
    outside string and character literals collapsed to one space: two
    sources that differ only in comments or layout give the same text.
    (Raw string literals and digit separators are not recognised; the kernel
    sources use neither.)"""
    out, i, n = [], 0, len(text)
    space = False
    while i < n:
        c = text[i]
        if c == "/" and i + 1 < n and text[i + 1] == "/":
            j = text.find("\n", i)
            i = n if j < 0 else j
            space = True
        elif c == "/" and i + 1 < n and text[i + 1] == "*":
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            space = True
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            if space and out:
                out.append(" ")
            space = False
            out.append(text[i:j + 1])
            i = j + 1
        elif c.isspace():
            space = True
            i += 1
        else:
            if space and out:
                out.append(" ")
            space = False
            out.append(c)
            i += 1
    return "".join(out)


def kernel_source_hash():
    """Hash of the fused kernel's code (comments and layout ignored), so an
    ncu summary stays attached to the code it measured."""
    h = hashlib.sha1()
    for f in ("k_compress.cuh", "k_compress.cu", "lamb1b_internal.cuh", "philox.cuh", "f32x2.cuh"):
        with open(os.path.join(ROOT, "communication_compressed_optimizer_gb300", "csrc", f)) as fh:
            h.update(code_tokens(fh.read()).encode())
    return h.hexdigest()[:12]


ISSUE_PEAK = 152 * 4 * 32 * 2070e6    # thread instructions per second (SMs x schedulers x lanes x clock)


def profile_summary(workload_name, variant="lamb", errors="f32"):
    """Path, relative to the repository, of the committed ncu summary of the
    fused kernel that this workload, method variant and error storage
    launch (each combination is its own kernel instantiation)."""
    tag = workload_name + ("_adam" if variant == "adam" else "") + ("_bf16err" if errors == "bf16" else "")
    return os.path.join("profiles", f"compress_kernel_{tag}.md")


def profiled_instructions(workload_name, variant="lamb", errors="f32"):
    """Thread instructions per launch of the fused kernel from the committed
    ncu summary (in-kernel gradient workloads), if taken on the current
    kernel source; else None."""
    path = os.path.join(ROOT, profile_summary(workload_name, variant, errors))
    if not os.path.exists(path):
        return None
    m = re.search(r"thread_inst_per_launch:\s*([0-9.eE+]+)\s+source_sha:\s*([0-9a-f]+)", open(path).read())
    if not m or m.group(2) != kernel_source_hash():
        return None
    return float(m.group(1))


def profiled_traffic(workload_name, variant="lamb", errors="f32"):
    """dram bytes per launch of the fused kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None.
    Returns (bytes or None, a description of where the figure comes from).
    It is not measured in this run: a DRAM-counter capture of the full-size
    workload is not taken under the profiler (the summary scales a small
    capture of the same kernel by the parameters processed)."""
    rel = profile_summary(workload_name, variant, errors)
    path = os.path.join(ROOT, rel)
    if not os.path.exists(path):
        return None, f"no ncu summary {rel}"
    text = open(path).read()
    m = re.search(r"traffic_per_launch_bytes:\s*([0-9.eE+]+)\s+source_sha:\s*([0-9a-f]+)", text)
    if not m:
        return None, f"{rel} records no traffic"
    if m.group(2) != kernel_source_hash():
        return None, f"{rel} was taken on kernel source {m.group(2)}, not the current {kernel_source_hash()}"
    return float(m.group(1)), (f"{rel}: ncu dram__bytes_read.sum + dram__bytes_write.sum of a smaller "
                               f"case of the same kernel, scaled by parameters to a full launch "
                               f"(kernel source {m.group(2)})")


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        self.out = os.path.join("/tmp", f"lamb1b_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.out, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.out):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.remove(self.out)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed helpers (one replica per rank, weak scaling)
# ---------------------------------------------------------------------------

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_throughput(local_seconds, units_per_rank, world):
    """Whole-job throughput of `world` replicas that each processed
    units_per_rank units in local_seconds: all units over the slowest rank's
    time (weak scaling).  Returns (units/s, slowest seconds)."""
    slowest = max_over_ranks(local_seconds, world)
    return world * units_per_rank / slowest, slowest


def host_memory_available():
    """MemAvailable of this host in bytes, or None where /proc/meminfo has none."""
    try:
        with open("/proc/meminfo") as fh:
            for line in fh:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def max_over_ranks(value, world):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample (baseline / reference arm)
# ---------------------------------------------------------------------------

def oracle_sample_rate(wl, seconds, max_steps=None, variant="lamb", errors="f32"):
    """Times the oracle's compression step on the leading chunks of the
    workload.  Returns (elements/s, description, steps, step times, sampled
    parameters, sampled chunks)."""
    import oracle
    C, W = wl.chunk, wl.W

    def make(nchunks):
        n = min(nchunks * C, wl.N)
        ends = wl.offsets + wl.numels
        frags = []
        for o, e in zip(wl.offsets, ends):
            if o >= n:
                break
            frags.append((int(o), int(min(e, n) - o)))
        x0 = workload.gen_params(wl, 0, n)
        o = oracle.Oracle([f[0] for f in frags], [f[1] for f in frags], W, C, wl.hp, x0,
                          variant=1 if variant == "adam" else 0, err_bf16=1 if errors == "bf16" else 0)
        o.v[:] = 1e-6
        o.freeze()
        g = np.empty((W, n), np.float32)
        for w in range(W):
            g[w] = workload.gen_grads_range(wl, 10, w, 0, n)
            if wl.grad == "bf16":
                g[w] = workload.bf16_round(g[w])
        return o, g, n

    o, g, n = make(8)
    t0 = time.perf_counter()
    o.compress_step(g)
    dt = time.perf_counter() - t0
    target = min(2.0, seconds / 5) if max_steps is None else max(0.05, seconds / max(1, max_steps))
    nchunks = int(max(1, min(wl.K, 8 * target / max(dt, 1e-6))))
    o, g, n = make(nchunks)
    times = []
    t_end = time.perf_counter() + seconds
    while time.perf_counter() < t_end and (max_steps is None or len(times) < max_steps):
        t0 = time.perf_counter()
        o.compress_step(g)
        times.append(time.perf_counter() - t0)
    rate = n / statistics.median(times)
    desc = (f"oracle compression step on the leading {n} parameters ({nchunks} chunks of "
            f"{C}, W={W}) of {wl.name}; median of {len(times)} steps")
    return rate, desc, len(times), times, n, nchunks


def variant_name(v):
    return "1-bit LAMB" if v == "lamb" else "1-bit Adam"


def cpu_info():
    model = ""
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return f"{os.uname().machine} {model}".strip(), os.cpu_count()


def run_reference(args, world, rank):
    if rank != 0:
        return
    wl = get_workload(args)
    total = max(30.0, 2.0 * (args.steps + args.warmup))
    per_step_budget = min(1.0, 120.0 / max(1, args.steps + args.warmup))
    rate, desc, n, times, n_params, n_chunks = oracle_sample_rate(
        wl, seconds=per_step_budget * (args.steps + args.warmup), max_steps=args.steps + args.warmup,
        variant=args.variant, errors=args.errors)
    timed = times[args.warmup:] or times
    ms = 1e3 * statistics.mean(timed)
    value = rate
    arch, ncpu = cpu_info()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": len(timed), "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "W": wl.W, "chunk": wl.chunk, "params": wl.N,
                   "tensors": wl.L, "grads": wl.grad, "variant": variant_name(args.variant),
                   "error_storage": args.errors,
                   # the oracle is timed on a bounded prefix of the table: the
                   # value is a rate (parameters per second), not a full step
                   "sampled_params": n_params, "sampled_chunks": n_chunks},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": desc, "host": arch, "host_cpus": ncpu},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    del total
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def live_copy_gbs(gib=2, reps=5):
    """Bandwidth of a plain device-to-device copy on this GPU, measured now
    (bytes read + bytes written per second, best of reps, 2 GiB each way).
    Context for the roofline fraction: the peak the fraction divides by is
    a single stored measurement, and GB300s differ by a few percent."""
    import torch
    n = (gib << 30) // 4
    src = torch.empty(n, dtype=torch.float32, device="cuda").fill_(1.0)
    dst = torch.empty_like(src)
    st = torch.cuda.current_stream()
    best = float("inf")
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(st)
        dst.copy_(src)
        b.record(st)
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b) / 1e3)
    del src, dst
    torch.cuda.empty_cache()
    return 2 * n * 4 / best / 1e9


def run_ours(args, world, rank, local):
    import torch

    import communication_compressed_optimizer_gb300 as pkg

    torch.cuda.set_device(local)
    wl = get_workload(args)
    N, W, C = wl.N, wl.W, wl.chunk
    layers = list(zip(wl.offsets.tolist(), wl.numels.tolist()))

    x = torch.empty(N, device="cuda")
    pkg.gen_params(x, 0, N, wl.param_std, wl.seed)
    opt = pkg.OneBitLamb(x, layers, W, C, **dict(wl.hp, variant=args.variant,
                                                 error_storage=args.errors))
    if wl.grad == "philox":
        g = pkg.PhiloxGrads(wl.seed, wl.layer_std, wl.layer_heavy, wl.heavy_scale)

        def regen(t):
            pass
        ld = 0
    else:
        q = 8 if wl.grad == "bf16" else 4
        ld = -(-N // q) * q
        g = torch.empty((W, ld), dtype=torch.int16 if wl.grad == "bf16" else torch.float32,
                        device="cuda")

        def regen(t):
            pkg.gen_grads(g, t, wl.seed, layers, wl.layer_std, None, wl.heavy_scale)

    def new_events():
        return [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    # warmup stage (LAMB), timed per step for information
    t = 0
    warm_ms, warm_kernel_ms, warm_layer_ms, warm_upd_ms = [], [], [], []
    n_warm_stage = wl.warmup_steps if args.warmup_stage_steps < 0 else args.warmup_stage_steps
    for _ in range(n_warm_stage):
        regen(t)
        ev = new_events()
        opt.set_trace_events(ev)
        opt.warmup_step(g)
        torch.cuda.synchronize()
        warm_ms.append(ev[0].elapsed_time(ev[3]))
        warm_kernel_ms.append(ev[0].elapsed_time(ev[1]))
        warm_layer_ms.append(ev[1].elapsed_time(ev[2]))
        warm_upd_ms.append(ev[2].elapsed_time(ev[3]))
        t += 1
    opt.freeze_variance()
    for _ in range(args.warmup):
        regen(t)
        opt.compress_step(g)
        t += 1
    opt.set_trace_events(None)
    torch.cuda.synchronize()
    barrier(world)

    # ---- timed region -------------------------------------------------------
    events = [new_events() for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        regen(t)
        opt.set_trace_events(events[i])
        opt.compress_step(g)
        t += 1
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    opt.set_trace_events(None)

    step_ms = [e[0].elapsed_time(e[3]) for e in events]
    kern_ms = [e[0].elapsed_time(e[1]) for e in events]
    factor_ms = [e[1].elapsed_time(e[2]) for e in events]
    upd_ms = [e[2].elapsed_time(e[3]) for e in events]
    value, total_s = aggregate_throughput(sum(step_ms) / 1e3, N * args.steps, world)
    ms_per_step = 1e3 * total_s / args.steps

    peak, peak_kind = measured_peaks()
    kb = fused_kernel_bytes(wl, args.variant, args.errors)
    k_avg = statistics.mean(kern_ms)
    achieved = kb / (k_avg / 1e3) / 1e9
    traffic, traffic_source = profiled_traffic(wl.name, args.variant, args.errors)
    copy_now = live_copy_gbs()
    roofline = {"bound": "hbm", "kernel": "k_compress (fused worker+server pass)",
                "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_source": peak_kind,
                "traffic": traffic, "traffic_source": traffic_source,
                "alg_bytes_per_launch": kb, "kernel_ms": k_avg,
                "live_copy_gbs": copy_now, "frac_of_live_copy": achieved / copy_now}
    if wl.grad == "philox":
        # gradients drawn in the kernel: bound by instruction issue, not HBM
        inst = profiled_instructions(wl.name, args.variant, args.errors)
        if inst is not None:
            t_ips = inst / (k_avg / 1e3)
            roofline = {"bound": "alu", "kernel": "k_compress (fused, in-kernel gradients)",
                        "achieved": t_ips / 1e12, "peak": ISSUE_PEAK / 1e12,
                        "unit": "T thread-inst/s", "frac": t_ips / ISSUE_PEAK,
                        "peak_source": "152 SMs x 4 schedulers x 32 lanes x 2070 MHz",
                        "traffic": traffic, "traffic_source": traffic_source,
                        "thread_inst_per_launch": inst, "kernel_ms": k_avg,
                        "hbm": {"achieved": achieved, "peak": peak, "unit": "GB/s",
                                "frac": achieved / peak, "alg_bytes_per_launch": kb,
                                "live_copy_gbs": copy_now}}

    # per-tensor coefficients after the timed steps: where the soft thresholds
    # and clip bounds are active
    sv = opt.state()
    r_now = sv["r_prev"].cpu().numpy()
    c_now = sv["c_cur"].cpu().numpy()
    cbar_now = sv["c_bar"].cpu().numpy()
    hp = wl.hp
    layer_stats = {
        "r_at_factor_max": int(np.sum(r_now >= np.float32(hp["factor_max"]))),
        "r_at_factor_min": int(np.sum(r_now <= np.float32(hp["factor_min"]))),
        "r_min": float(r_now.min()), "r_max": float(r_now.max()),
        "c_min": float(c_now.min()), "c_max": float(c_now.max()),
        "c_bar_at_clip": int(np.sum((cbar_now <= np.float32(hp["coeff_min"]))
                                    | (cbar_now >= np.float32(hp["coeff_max"])))),
        "tensors": int(len(r_now))}

    # ---- end to end through the public API with host buffers ----------------
    e2e = None
    if not args.no_e2e and args.e2e_steps > 0:
        # every local rank pins one step of gradients in host memory: never
        # more than half of what the host has available
        h2d = 0 if wl.grad == "philox" else W * ld * grad_bytes(wl)
        local = int(os.environ.get("LOCAL_WORLD_SIZE", world))
        avail = host_memory_available()
        fits = h2d == 0 or (avail is not None and local * h2d <= 0.5 * avail)
        if max_over_ranks(0.0 if fits else 1.0, world) == 0.0:
            e2e = run_e2e(args, opt, wl, g, regen, t, ld)
            slowest = max_over_ranks(e2e.pop("_seconds"), world)
            e2e["value"] = world * N * args.e2e_steps / slowest
            e2e["ms_per_step"] = 1e3 * slowest / args.e2e_steps
            t += args.e2e_steps + 1
        else:
            e2e = {"value": None, "unit": UNIT,
                   "skipped": "host memory: %d local ranks x %.1f GB of pinned gradients exceed half of "
                              "the %.0f GB available" % (local, h2d / 1e9, (avail or 0) / 1e9)}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl.name, "W": W, "chunk": C, "params": N, "tensors": wl.L,
                   "grads": wl.grad, "variant": variant_name(args.variant),
                   "error_storage": args.errors,
                   "parallelism": f"replicas{world}",
                   "l2": "inputs larger than L2 (each step moves %.1f GB); gradients regenerated "
                         "on the device between timed steps" % (step_bytes(wl, args.variant, args.errors) / 1e9),
                   "timing": "CUDA events on the launching stream around each step"},
        "roofline": roofline,
        "step": {"alg_bytes": step_bytes(wl, args.variant, args.errors), "hbm_gbs": step_bytes(wl, args.variant, args.errors) / (ms_per_step / 1e3) / 1e9,
                 "frac_of_peak": step_bytes(wl, args.variant, args.errors) / (ms_per_step / 1e3) / 1e9 / peak,
                 "kernel_ms": {"compress": k_avg, "factor": statistics.mean(factor_ms),
                               "update": statistics.mean(upd_ms)},
                 # the step's other streaming kernel, against the same peak
                 "update_gbs": update_kernel_bytes(wl) / (statistics.mean(upd_ms) / 1e3) / 1e9,
                 "update_frac_of_peak": update_kernel_bytes(wl) / (statistics.mean(upd_ms) / 1e3) / 1e9 / peak,
                 "ms_p10": float(np.percentile(step_ms, 10)),
                 "ms_p50": float(np.percentile(step_ms, 50)),
                 "ms_p90": float(np.percentile(step_ms, 90)),
                 "worker_elements_per_s": W * value, "wall_s": wall},
        "warmup_stage": (warmup_stage_line(wl, args.variant, N, peak, warm_ms, warm_kernel_ms,
                                           warm_layer_ms, warm_upd_ms) if warm_ms else None),
        "gpu_launches": (2 if args.variant == "adam" else 3) * args.steps,
        "layer_stats": layer_stats,
        "clocks": clocks,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, desc, n, _, _, _ = oracle_sample_rate(wl, seconds=args.cpu_seconds, variant=args.variant,
                                                    errors=args.errors)
        arch, ncpu = cpu_info()
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": desc, "host": arch, "host_cpus": ncpu}
    if rank == 0:
        print(json.dumps(line), flush=True)
    opt.close()


def run_e2e(args, opt, wl, g, regen, t, ld):
    """Same metric through the public API with host buffers.  Stored
    gradients: every step is one lamb1b_compress_step_host call, which copies
    that step's gradients from pinned host memory into a staging buffer (two
    used in turn; the copy on its own stream, overlapping the previous step's
    kernels), runs the step and reads the server's compressed message (sign
    words and chunk scales) back into pinned host memory.  In-kernel
    gradients have no host input: the step plus the same read-back."""
    import torch
    nw, K = -(-wl.N // 32), -(-wl.N // wl.chunk)
    out_w = torch.empty(nw, dtype=torch.int32, pin_memory=True)
    out_s = torch.empty(K, dtype=torch.float32, pin_memory=True)
    d2h = 4 * nw + 4 * K
    compute = torch.cuda.current_stream()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if wl.grad == "philox":
        st = opt.state(sync=False)
        words, scales = st["signs_s"][:nw], st["scale_s"][:K]
        torch.cuda.synchronize()
        s0.record(compute)
        for _ in range(args.e2e_steps):
            opt.compress_step(g)
            out_w.copy_(words, non_blocking=True)
            out_s.copy_(scales, non_blocking=True)
        s1.record(compute)
        torch.cuda.synchronize()
        h2d = 0
        extra = {"path": "lamb1b_compress_step (in-kernel gradients) + read-back of the server message"}
    else:
        regen(t)
        host = torch.empty(g.shape, dtype=g.dtype, pin_memory=True)
        host.copy_(g)
        h2d = g.numel() * g.element_size()
        bufs = [g, torch.empty_like(g)]
        copy = torch.cuda.Stream()
        # one copy with nothing else running, for comparison
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        with torch.cuda.stream(copy):
            a0.record(copy)
            bufs[1].copy_(host, non_blocking=True)
            a1.record(copy)
        torch.cuda.synchronize()
        alone_ms = a0.elapsed_time(a1)
        # untimed: one call per staging buffer, so that the timed calls find
        # both buffers known to the context (a buffer's first copy waits for
        # everything already on the step stream)
        for i in range(2):
            opt.compress_step_host(host, bufs[i], out_w, out_s, stream=compute, copy_stream=copy)
        torch.cuda.synchronize()
        # per-step end times on the step stream
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.e2e_steps)]
        s0.record(compute)
        copy.wait_event(s0)
        for i in range(args.e2e_steps):
            opt.compress_step_host(host, bufs[i % 2], out_w, out_s, stream=compute, copy_stream=copy)
            ends[i].record(compute)
        s1.record(compute)
        torch.cuda.synchronize()
        step_ms = [s0.elapsed_time(ends[0])] + [ends[i - 1].elapsed_time(ends[i])
                                                 for i in range(1, args.e2e_steps)]
        extra = {"path": "lamb1b_compress_step_host: pinned host gradients -> staging buffers used in "
                         "turn on a copy stream, overlapping the previous step's kernels; server message "
                         "read back to pinned host memory",
                 "step_ms": [round(x, 3) for x in step_ms],
                 "copy_alone_gbs": h2d / (alone_ms / 1e3) / 1e9}
        del bufs[1]
    sec = s0.elapsed_time(s1) / 1e3
    out = {"value": wl.N * args.e2e_steps / sec, "_seconds": sec, "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
           "ms_per_step": 1e3 * sec / args.e2e_steps,
           "h2d_gbs": (h2d / (sec / args.e2e_steps) / 1e9) if h2d else None}
    out.update(extra)
    return out


def main():
    args = parse_args()
    if args.impl == "reference":
        # the CPU oracle needs no collective: rank 0 alone runs it, the others
        # exit without joining a process group
        run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
        return
    world, rank, local = dist_setup(args)
    run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
