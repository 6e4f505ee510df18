"""Benchmark: effective FP32 TFLOPS of the emulated GEMMs on PET-shaped layers.

One step = the hot path over one batch: the forward GEMM of a PET-like linear
layer, Y = X W^T + b (M = 6144 tokens = 192 atoms x 32 neighbours, K = 256,
N = 1024), and its input-gradient GEMM dX = dY W, both through the C ABI
(emu_linear_fwd, emu_linear_bwd_input).  Effective FLOPs = 2 M N K per GEMM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--mode bf16x9|tf32x3]
                    [--workload pet_small|pet_large|wide_l1|wide_l2] [--impl ours|reference]

Prints one JSON line (rank 0).  Inputs are synthetic (seeded; X ~ N(0,1),
W ~ N(0,1/K), b ~ N(0,0.01), dY ~ N(0,1)).  The L2 cache (129 MB) is flushed
between timed steps by writing a 256 MB buffer; step times are CUDA-event
device times of the two GEMM launches on the launching stream.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "effective FP32 TFLOPS (BF16x9 GEMM, PET shapes) and % of BF16-peak/9 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--mode", default="bf16x9", choices=["bf16x9", "tf32x3", "tf32x1", "bf16x6"])
    ap.add_argument("--workload", default="pet_small", choices=["pet_small", "pet_large", "wide_l1", "wide_l2"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-comparators", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads and modes reported under extras.workloads")
    ap.add_argument("--rows", type=int, default=0,
                    help="replace the workload's M (token rows) by this many, for profiler captures of a "
                         "smaller case of the same kernel; the JSON line names the changed workload")
    return ap.parse_args()


def shape_of(name, rows=0):
    import dataclasses
    from fp32_emulated_gemm_gb300 import workloads as W
    s = {"pet_small": W.PET_SMALL, "pet_large": W.PET_LARGE, "wide_l1": W.WIDE_L1, "wide_l2": W.WIDE_L2}[name]
    return dataclasses.replace(s, M=rows) if rows > 0 else s


def config_id(name):
    return {"pet_small": 2, "pet_large": 3, "wide_l1": 4, "wide_l2": 4}[name]


def max_over_ranks(x, world, device):
    """The largest of every rank's x (the slowest replica sets the job's
    time); x itself on one process."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank_step, world, step_ms):
    """Replicas: every rank does one step's work in the (slowest) step time."""
    return world * flops_per_rank_step / (step_ms * 1e-3) / 1e12


def step_flops(s):
    return 2 * (2.0 * s.M * s.N * s.K)  # forward + input gradient


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
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
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def host_info():
    """The CPU this runs on: model name (x86 'model name', Arm implementer /
    part ids) and the cores this process may use."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            txt = f.read()
        for key in ("model name", "Model", "CPU part"):
            for line in txt.splitlines():
                if line.lower().startswith(key.lower()):
                    model = (model + ", " if model else "") + line.split(":", 1)[1].strip()
                    break
            if model and key == "model name":
                break
    except OSError:
        pass
    import platform
    usable = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"model": model or platform.processor() or platform.machine(), "machine": platform.machine(),
            "nproc": usable, "cpu_count": os.cpu_count()}


_ONE_CORE_CODE = r"""
import json, sys, time
sys.path.insert(0, %r)
import oracle
from fp32_emulated_gemm_gb300 import workloads as W
s = W.PET_SMALL
X, Wt, b, dY = W.linear_inputs(s, W.CONFIG_ID["pet_small"], rows=%d)
out = {"threads": oracle.num_threads()}
for mode in ("bf16x9", "tf32x3"):
    t = time.perf_counter()
    oracle.gemm_emulated(oracle.Problem(X, Wt, transB=True, bias=b), mode)
    oracle.gemm_emulated(oracle.Problem(dY, Wt), mode)
    out[mode] = time.perf_counter() - t
print(json.dumps(out))
"""


def cpu_protocol():
    """The oracle's timing protocol on this host: the PET-small step (forward
    + input gradient) and the tiny problem in full on all cores; the wide
    layers on the deterministic row sample of their parity tests (every
    128th row plus the first and last 64), extrapolated to all rows and
    labelled so; and the PET-small
    step on a 256-row sample on one core (a child process with
    OMP_NUM_THREADS=1).  Seconds per step, both modes."""
    import oracle
    from fp32_emulated_gemm_gb300 import workloads as W
    res = {"host": host_info(), "threads_all": oracle.num_threads()}
    A, B, Cold = W.tiny_inputs()
    for mode in ("bf16x9", "tf32x3"):
        t = time.perf_counter()
        oracle.gemm_emulated(oracle.Problem(A, B, beta=1.0, C_old=Cold), mode)
        res.setdefault("tiny_full_s", {})[mode] = time.perf_counter() - t
    s = W.PET_SMALL
    X, Wt, b, dY = W.linear_inputs(s, W.CONFIG_ID["pet_small"])
    for mode in ("bf16x9", "tf32x3"):
        t = time.perf_counter()
        oracle.gemm_emulated(oracle.Problem(X, Wt, transB=True, bias=b), mode)
        oracle.gemm_emulated(oracle.Problem(dY, Wt), mode)
        dt = time.perf_counter() - t
        res.setdefault("pet_small_full_step_s", {})[mode] = dt
    for lname, shape in (("wide_l1", W.WIDE_L1), ("wide_l2", W.WIDE_L2)):
        rows = W.sample_rows(shape.M, every=128, edge=64)
        X, Wt, b, dY = W.linear_inputs(shape, W.CONFIG_ID["wide"])
        for mode in ("bf16x9", "tf32x3"):
            t = time.perf_counter()
            oracle.gemm_emulated(oracle.Problem(X, Wt, transB=True, bias=b), mode, rows)
            oracle.gemm_emulated(oracle.Problem(dY, Wt), mode, rows)
            dt = time.perf_counter() - t
            res.setdefault(f"{lname}_sampled", {})[mode] = {
                "rows": int(rows.size), "of": shape.M, "sample_s": dt,
                "full_step_s_extrapolated": dt * shape.M / rows.size}
    r1 = 256
    try:
        out = subprocess.run([sys.executable, "-c", _ONE_CORE_CODE % (ROOT, r1)], capture_output=True,
                             text=True, timeout=300, env=dict(os.environ, OMP_NUM_THREADS="1"))
        one = json.loads(out.stdout.strip().splitlines()[-1])
        res["one_core"] = {"threads": one["threads"], "sample": f"PET-small step on the first {r1} of {s.M} rows",
                           **{m: {"sample_s": one[m], "full_step_s_extrapolated": one[m] * s.M / r1}
                              for m in ("bf16x9", "tf32x3")}}
    except Exception as exc:  # reported, not fatal
        res["one_core"] = {"unavailable": str(exc)[:200]}
    return res


def cpu_baseline(shape, mode, target_s=10.0):
    """The CPU oracle on a bounded row sample of the same step (forward + input
    gradient on the first r rows), timed on this host's cores."""
    import oracle
    from fp32_emulated_gemm_gb300 import workloads as W
    oracle.build()
    X, Wt, b, dY = W.linear_inputs(shape, config_id_for_shape(shape), rows=min(shape.M, 4096))

    def run(r):
        t = time.perf_counter()
        oracle.gemm_emulated(oracle.Problem(X[:r], Wt, transB=True, bias=b), mode)
        oracle.gemm_emulated(oracle.Problem(dY[:r], Wt), mode)
        return time.perf_counter() - t

    r = 16
    dt = run(r)
    while dt < target_s / 4 and r < X.shape[0]:
        r = min(X.shape[0], r * 4)
        dt = run(r)
    flops = 2 * (2.0 * r * shape.N * shape.K)
    # the oracle's other functions on the same sample: rows per second and
    # the full workload's time extrapolated from it
    funcs = {}
    for name, fn in (("gemm_f64", oracle.gemm_f64), ("sgemm_f32", oracle.sgemm_f32),
                     ("gemm_bf16x9", oracle.gemm_bf16x9), ("gemm_tf32x3", oracle.gemm_tf32x3)):
        t = time.perf_counter()
        fn(oracle.Problem(X[:r], Wt, transB=True, bias=b))
        fn(oracle.Problem(dY[:r], Wt))
        ft = time.perf_counter() - t
        funcs[name] = {"rows_per_s": r / ft, "full_step_s_extrapolated": ft * shape.M / r}
    return {"value": flops / dt / 1e12, "unit": "TFLOPS", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"forward + input gradient on the first {r} of {shape.M} rows ({mode}), {dt:.2f} s",
            "functions": funcs, "protocol": cpu_protocol()}


def config_id_for_shape(shape):
    return {"pet_small": 2, "pet_large": 3, "wide_l1": 4, "wide_l2": 4}[shape.name]


def run_reference(args, world, rank):
    """--impl reference: the CPU oracle (as it stands) on this host's cores,
    one bounded row sample of the workload per step."""
    if rank != 0:
        return
    import oracle
    from fp32_emulated_gemm_gb300 import workloads as W
    oracle.build()
    s = shape_of(args.workload, args.rows)
    X, Wt, b, dY = W.linear_inputs(s, config_id(args.workload), rows=64)
    r = 8  # rows per step: keeps --steps K runs within minutes

    def step():
        oracle.gemm_emulated(oracle.Problem(X[:r], Wt, transB=True, bias=b), args.mode)
        oracle.gemm_emulated(oracle.Problem(dY[:r], Wt), args.mode)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t
    flops = 2 * (2.0 * r * s.N * s.K) * args.steps
    v = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(args, s),
        "cpu_baseline": {"value": v, "unit": "TFLOPS", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{r} of {s.M} rows of the forward and input-gradient GEMMs per step"},
        "e2e": {"value": v, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(args, s):
    return {"workload": f"{s.name}: Y = X W^T + b and dX = dY W, M={s.M} K={s.K} N={s.N}",
            "mode": args.mode, "M": s.M, "K": s.K, "N": s.N, "gemms_per_step": 2,
            "l2": "flushed between timed steps (256 MB write)", "parallelism": f"replicas x{args.gpus}"}


def main():
    args = parse()
    world, rank, local = dist_init(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import numpy as np
    import torch
    import fp32_emulated_gemm_gb300 as emu
    from fp32_emulated_gemm_gb300 import build as emu_build
    from fp32_emulated_gemm_gb300 import workloads as W

    emu_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    s = shape_of(args.workload, args.rows)
    mode = emu.MODES[args.mode]
    X, Wt, b, dY = W.linear_inputs(s, config_id(args.workload))
    Xd, Wd, bd, dYd = (torch.from_numpy(a).to(dev) for a in (X, Wt, b, dY))
    Yd = torch.empty((s.M, s.N), device=dev)
    dXd = torch.empty((s.M, s.K), device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    def fwd():
        emu.emu_linear_fwd(mode, s.M, s.N, s.K, Xd, Wd, bd, Yd, sp)

    def bwd():
        emu.emu_linear_bwd_input(mode, s.M, s.N, s.K, dYd, Wd, dXd, sp)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1.0)
        fwd()
        bwd()
    st = emu.emu_stream_check(sp)
    if st != 0:
        raise RuntimeError(emu.emu_status_string(st))

    K = args.steps
    # one event pair per step: the two launches run back to back, as in a
    # model (the second may start its set-up while the first finishes)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    sampler = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.15)
    t_wall = time.perf_counter()
    for i in range(K):
        flush.fill_(float(i & 7))
        ev[i][0].record(stream)
        fwd()
        bwd()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    st = emu.emu_stream_check(sp)
    if st != 0:
        raise RuntimeError(emu.emu_status_string(st))
    step_ms = sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(K)) / K
    fwd_ms, bwd_ms = isolated_launch_ms(stream, flush, fwd, bwd, min(K, 200))
    step_ms = max_over_ranks(step_ms, world, dev)
    flops = step_flops(s)
    value = whole_job_tflops(flops, world, step_ms)

    peaks, peak_kind = load_peaks()
    peak = peaks["bf16_tflops"] / TENSOR_UNITS[args.mode]
    # dominant kernel: the emulated-GEMM kernel (both launches of a step);
    # algorithmic work per launch = 2 M N K effective FLOPs, over the average
    # duration of a launch timed alone (events on both sides of it, no
    # overlap with its neighbour); the step-based figure, which credits the
    # overlap of the two launches, is reported beside it
    achieved = (flops / 2) / (0.5 * (fwd_ms + bwd_ms) * 1e-3) / 1e12
    achieved_step = (flops / 2) / ((step_ms / 2) * 1e-3) / 1e12
    traffic = load_traffic(args)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(emu, mode, s, X, Wt, b, dY, dev, stream, n=max(5, min(K, 50)))
        e2e["ms"] = max_over_ranks(e2e["ms"], world, dev)
        e2e = {"value": whole_job_tflops(flops, world, e2e["ms"]), "unit": "TFLOPS",
               "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"]}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": args.mode, "data": "synthetic",
        "config": workload_config(args, s),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} bf16 dense burst / {TENSOR_UNITS[args.mode]:g}",
                     "kernel": f"emu_gemm_kernel<{args.mode}>",
                     "launch_ms": 0.5 * (fwd_ms + bwd_ms),
                     "isolated_fwd_ms": fwd_ms, "isolated_bwd_ms": bwd_ms,
                     "achieved_step": achieved_step, "frac_step": achieved_step / peak,
                     "step_launch_ms": step_ms / 2},
        "gpu_launches": launches_per_step(emu, args.mode, s) * K,
        "wall_s_timed_region": wall,
    }
    if clocks:
        line["clocks"] = clocks
    if e2e:
        line["e2e"] = e2e
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(s, args.mode)
    if not args.no_comparators:
        line["comparators"] = cublas_comparators(s)
        line["extras"] = extra_passes(emu, mode, s, Xd, dYd, flush, stream, fwd, bwd, peak)
        if not args.no_workloads and args.rows == 0:
            line["extras"]["workloads"] = other_workloads(emu, args, peaks, peak_kind, dev, stream, flush)
    print(json.dumps(line), flush=True)


# tensor work per effective FLOP, in BF16-rate units (TF32 runs at half rate)
TENSOR_UNITS = {"bf16x9": 9.0, "bf16x6": 6.0, "tf32x3": 6.0, "tf32x1": 2.0}

# Beside the headline (PET-small, BF16x9), the same measurement on the other
# PET-shaped workloads and in the other mode.
OTHER_WORKLOADS = [("pet_small", "tf32x3"), ("pet_large", "bf16x9"), ("pet_large", "tf32x3"),
                   ("wide_l1", "bf16x9"), ("wide_l1", "tf32x3"), ("wide_l2", "bf16x9"), ("wide_l2", "tf32x3")]


def device_linear_inputs(s, config, dev):
    """The workload's inputs drawn on the device (seeded torch generators,
    one per tensor, seed 100 config + tensor id; X ~ N(0,1), W ~ N(0,1/K),
    b ~ N(0,0.01), dY ~ N(0,1)): the large workloads' gigabytes need no host
    draw or copy.  Same distributions as workloads.linear_inputs."""
    import torch

    def normal(shape, std, tensor_id):
        g = torch.Generator(device=dev)
        g.manual_seed(100 * config + tensor_id)
        return torch.randn(shape, generator=g, device=dev).mul_(std)

    return (normal((s.M, s.K), 1.0, 0), normal((s.N, s.K), s.K ** -0.5, 1), normal((s.N,), 0.1, 2),
            normal((s.M, s.N), 1.0, 3))


def other_workloads(emu, args, peaks, peak_kind, dev, stream, flush):
    """Each (workload, mode) of OTHER_WORKLOADS timed like the headline: the
    step (forward + input gradient between one event pair, L2 flushed before
    it) and each launch alone; effective TFLOPS and the fraction of the
    measured BF16 peak over the mode's tensor work, both from the step and
    from the launches timed alone (the kernel's own duration, no overlap)."""
    import torch
    out = {}
    sp = stream.cuda_stream
    for name, mode_name in OTHER_WORKLOADS:
        s = shape_of(name)
        mode = emu.MODES[mode_name]
        X, Wt, b, dY = device_linear_inputs(s, config_id(name), dev)
        Y = torch.empty((s.M, s.N), device=dev)
        dX = torch.empty((s.M, s.K), device=dev)

        def fwd():
            emu.emu_linear_fwd(mode, s.M, s.N, s.K, X, Wt, b, Y, sp)

        def bwd():
            emu.emu_linear_bwd_input(mode, s.M, s.N, s.K, dY, Wt, dX, sp)

        flops = step_flops(s)
        K = 20 if s.M > 100000 else 100
        for _ in range(3):
            flush.fill_(1.0)
            fwd()
            bwd()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        for i in range(K):
            flush.fill_(float(i & 7))
            ev[i][0].record(stream)
            fwd()
            bwd()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        st = emu.emu_stream_check(sp)
        if st != 0:
            raise RuntimeError(f"{name} {mode_name}: {emu.emu_status_string(st)}")
        step_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
        f_ms, b_ms = isolated_launch_ms(stream, flush, fwd, bwd, K)
        peak = peaks["bf16_tflops"] / TENSOR_UNITS[mode_name]
        iso = (flops / 2) / (0.5 * (f_ms + b_ms) * 1e-3) / 1e12
        val = flops / (step_ms * 1e-3) / 1e12
        out[f"{name}_{mode_name}"] = {
            "workload": f"{name}: M={s.M} K={s.K} N={s.N}, forward + input gradient", "mode": mode_name,
            "steps": K, "ms_per_step": step_ms, "value": val, "unit": "TFLOPS", "frac_step": val / peak,
            "isolated_fwd_ms": f_ms, "isolated_bwd_ms": b_ms, "achieved_isolated": iso, "frac_isolated": iso / peak,
            "peak": peak, "peak_source": f"{peak_kind} bf16 dense burst / {TENSOR_UNITS[mode_name]:g}",
            "gpu_launches_per_step": launches_per_step(emu, mode_name, s),
            "l2": "flushed before every step (256 MB write)", "inputs": "drawn on the device, seeded"}
        del X, Wt, b, dY, Y, dX
        torch.cuda.empty_cache()
    return out


def launches_per_step(emu, mode, s):
    """Kernels one step launches: one per GEMM, plus, in the TF32 modes, the
    library's split of op(B) ahead of a product whose op(A) spans four or
    more 256-row tiles (unless EMU_AUTOPACK=0)."""
    n = 0
    for (m, n_out, k) in ((s.M, s.N, s.K), (s.M, s.K, s.N)):   # forward, input gradient
        n += 1
        if (mode in ("tf32x3", "tf32x1") and os.environ.get("EMU_AUTOPACK", "1") != "0"
                and -(-m // 256) >= 4 and emu.emu_pack_bytes(mode, n_out, k) <= (1 << 30)):
            n += 1
    return n


def extra_passes(emu, mode, s, Xd, dYd, flush, stream, fwd, bwd, peak, n=100):
    """Context beside the headline, after the timed region: the emulated
    weight gradient dW = dY^T X of the same layer (one launch, L2 flushed
    before it), and the step with L2 warm (50 steps back to back between one
    event pair: inputs and outputs stay in L2, as in steady-state inference)."""
    import torch
    sp = stream.cuda_stream
    dW = torch.empty((s.N, s.K), device=Xd.device)

    def wgrad():
        emu.emu_linear_bwd_weight(mode, s.M, s.N, s.K, dYd, Xd, 0.0, dW, sp)

    for _ in range(3):
        wgrad()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for i in range(n):
        flush.fill_(1.0)
        ev[i][0].record(stream)
        wgrad()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wg_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / n
    wg_tf = 2.0 * s.M * s.N * s.K / (wg_ms * 1e-3) / 1e12
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(5):
        fwd()
        bwd()
    e0.record(stream)
    warm = 50
    for _ in range(warm):
        fwd()
        bwd()
    e1.record(stream)
    torch.cuda.synchronize()
    st = emu.emu_stream_check(sp)
    if st != 0:
        raise RuntimeError(emu.emu_status_string(st))
    warm_ms = e0.elapsed_time(e1) / warm
    warm_tf = step_flops(s) / (warm_ms * 1e-3) / 1e12
    return {"weight_grad": {"value": wg_tf, "unit": "TFLOPS", "ms": wg_ms, "frac": wg_tf / peak,
                            "pass": f"dW[{s.N},{s.K}] = dY^T X, contraction over M={s.M}, L2 flushed"},
            "warm_step": {"value": warm_tf, "unit": "TFLOPS", "ms_per_step": warm_ms, "frac": warm_tf / peak,
                          "l2": "warm (50 steps back to back)"}}


def isolated_launch_ms(stream, flush, fwd, bwd, n):
    """Each launch timed alone (an event on either side of it, so the two do
    not overlap), after the timed region: the per-pass split of a step."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    for i in range(n):
        flush.fill_(1.0)
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        ev[i][2].record(stream)
        bwd()
        ev[i][3].record(stream)
    torch.cuda.synchronize()
    f = sum(e[0].elapsed_time(e[1]) for e in ev) / n
    b = sum(e[2].elapsed_time(e[3]) for e in ev) / n
    return f, b


def cublas_comparators(shape, steps=200):
    """Same step through torch.matmul on the same GPU: native FP32 SGEMM
    (TF32 off) and cuBLAS's own BF16x9 path (CUBLAS_EMULATE_SINGLE_PRECISION=1,
    set before cuBLAS loads, so it runs in a child process).  Context only."""
    out = {}
    code = r"""
import json, os, sys, torch
M, K, N, steps = %d, %d, %d, %d
torch.backends.cuda.matmul.allow_tf32 = False
dev = torch.device('cuda')
X = torch.randn(M, K, device=dev); W = torch.randn(N, K, device=dev) / K ** 0.5
b = torch.randn(N, device=dev) * 0.1; dY = torch.randn(M, N, device=dev)
flush = torch.empty(64 * 1024 * 1024, device=dev)
def step():
    torch.addmm(b, X, W.t()); dY.mm(W)
for _ in range(10): step()
torch.cuda.synchronize()
tot = 0.0
for _ in range(steps):
    flush.fill_(1.0)
    e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
    e0.record(); step(); e1.record(); torch.cuda.synchronize(); tot += e0.elapsed_time(e1)
print(json.dumps({"ms": tot / steps}))
""" % (shape.M, shape.K, shape.N, steps)
    for name, env in (("cublas_sgemm_native", {}), ("cublas_bf16x9_emulated", {"CUBLAS_EMULATE_SINGLE_PRECISION": "1"})):
        try:
            r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300,
                               env=dict(os.environ, **env))
            ms = json.loads(r.stdout.strip().splitlines()[-1])["ms"]
            out[name] = {"value": step_flops(shape) / (ms * 1e-3) / 1e12, "unit": "TFLOPS", "ms_per_step": ms}
        except Exception as exc:  # reported, not fatal
            out[name] = {"unavailable": str(exc)[:200]}
    return out


def kernel_source_hash():
    """sha256 over the CUDA sources of the library (what an ncu capture measured)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp32_emulated_gemm_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def load_traffic(args):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary for this workload, or None when no capture exists or the kernel
    sources changed since the counters were taken."""
    if args.rows:
        return None  # the committed counters are for the full workload
    path = os.path.join(ROOT, "profiles", f"traffic_{args.workload}_{args.mode}.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("kernel_source_sha256") != kernel_source_hash():
            return None
        return d.get("dram_bytes_per_launch")
    except Exception:
        return None


def run_e2e(emu, mode, s, X, Wt, b, dY, dev, stream, n):
    """Same step through the public API from pinned host buffers: every step
    copies its inputs (X, W, b, dY) host to device, runs both GEMMs and copies
    both results (Y, dX) device to host.  As an application would, the copies
    run on their own streams (one per direction) and overlap the GEMMs of the
    same and the neighbouring steps: the forward waits only for X, W and b,
    the input gradient for dY, and each result leaves as soon as it is done;
    device buffers alternate between two sets so that a step's inputs can
    arrive while the previous step still computes."""
    import torch
    hX, hW, hb, hdY = (torch.from_numpy(a).pin_memory() for a in (X, Wt, b, dY))
    hY = [torch.empty((s.M, s.N)).pin_memory() for _ in range(2)]
    hdX = [torch.empty((s.M, s.K)).pin_memory() for _ in range(2)]
    sets = [dict(X=torch.empty_like(hX, device=dev), W=torch.empty_like(hW, device=dev),
                 b=torch.empty_like(hb, device=dev), dY=torch.empty_like(hdY, device=dev),
                 Y=torch.empty((s.M, s.N), device=dev), dX=torch.empty((s.M, s.K), device=dev)) for _ in range(2)]
    h2d = torch.cuda.Stream(dev)
    d2h = torch.cuda.Stream(dev)
    comp = stream
    E = lambda: torch.cuda.Event()
    freed = [[E(), E()] for _ in range(2)]   # per set: inputs consumed, outputs copied out
    state = {"i": 0}

    def step():
        k = state["i"] % 2
        d = sets[k]
        fwd_in, bwd_in, y_done, dx_done = E(), E(), E(), E()
        with torch.cuda.stream(h2d):
            h2d.wait_event(freed[k][0])              # the set's previous inputs are consumed
            d["X"].copy_(hX, non_blocking=True)
            d["W"].copy_(hW, non_blocking=True)
            d["b"].copy_(hb, non_blocking=True)
            fwd_in.record(h2d)
            d["dY"].copy_(hdY, non_blocking=True)
            bwd_in.record(h2d)
        comp.wait_event(fwd_in)
        comp.wait_event(freed[k][1])                 # the set's previous results have left
        emu.emu_linear_fwd(mode, s.M, s.N, s.K, d["X"], d["W"], d["b"], d["Y"], comp.cuda_stream)
        y_done.record(comp)
        comp.wait_event(bwd_in)
        emu.emu_linear_bwd_input(mode, s.M, s.N, s.K, d["dY"], d["W"], d["dX"], comp.cuda_stream)
        dx_done.record(comp)
        freed[k][0] = E()
        freed[k][0].record(comp)
        with torch.cuda.stream(d2h):
            d2h.wait_event(y_done)
            hY[k].copy_(d["Y"], non_blocking=True)
            d2h.wait_event(dx_done)
            hdX[k].copy_(d["dX"], non_blocking=True)
            freed[k][1] = E()
            freed[k][1].record(d2h)
        state["i"] += 1

    for k in range(2):
        freed[k][0].record(comp)
        freed[k][1].record(comp)
    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    h2d.wait_event(e0)
    d2h.wait_event(e0)
    for _ in range(n):
        step()
    done = [E(), E()]
    done[0].record(h2d)
    done[1].record(d2h)
    comp.wait_event(done[0])
    comp.wait_event(done[1])
    e1.record(comp)
    torch.cuda.synchronize(dev)
    h2d_bytes = sum(t.numel() * 4 for t in (hX, hW, hb, hdY))
    d2h_bytes = (hY[0].numel() + hdX[0].numel()) * 4
    return {"ms": e0.elapsed_time(e1) / n, "h2d": h2d_bytes, "d2h": d2h_bytes}


if __name__ == "__main__":
    main()
