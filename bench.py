#!/usr/bin/env python3
"""Benchmark of the MXFP4 Wgrad hot path on one GB300.

Metric: MXFP4 Wgrad TFLOP/s including the Hadamard rotation and quantisation,
2*N*K*T / step time, on the largest single-GPU Llama-3.1-8B Wgrad shape, the
FFN down_proj (T = 8192 tokens, dY [8192, 4096], X [8192, 14336] -> dW
[4096, 14336] fp32), deterministic block Hadamard of 32 along T,
round-to-nearest-even.  The attention o_proj shape (N = K = 4096) is timed
beside it.  Inputs are synthetic (seeded; Student-t(3) gradients with std
1e-3; SiLU(g)*u activations for down_proj, N(0,1) with 1% x20 outlier
channels for o_proj) and resident in HBM when the timed region starts.

One step = the two launches of the hot path through the C ABI:
mx_quantize_pair(dY, X) (both operands rotated and encoded in one launch) and
mx_gemm.  L2 is flushed (512 MB write)
before every timed step, outside the events.  `e2e` repeats the step through
mx_linear_wgrad with pinned HOST buffers, the H2D/D2H copies inside the
timed region.  The reference arm (--impl reference) times the CPU oracle on
a bounded sample of the same workload.

Multi-GPU: the path runs as independent replicas (weak scaling); under
torchrun every rank times its own replica and rank 0 reports
sum(units) / max(time).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MXFP4 Wgrad TFLOPS incl. Hadamard+quant, Llama-3.1-8B shapes; % FP4 peak"
WORKLOADS = {
    # name: (config key, T, N, K)
    "o_proj": ("o_proj", 8192, 4096, 4096),
    "down_proj": ("down_proj", 8192, 4096, 14336),
}
NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25      # nominal dense ratio (recipe table)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(name: str) -> str:
    with open(os.path.join(ROOT, "mxfp4_precision_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def load_traffic():
    """DRAM bytes per launch from committed ncu summaries (profiles/traffic.txt):
    lines `kernel source_hash workload bytes`.  Ignored when the kernel source
    changed since the capture."""
    out = {}
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return out
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if len(line) == 4:
                out[(line[0], line[2])] = (line[1], float(line[3]))
    return out


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx_, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx_.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx_),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(local_total_ms: float, steps: int, units_per_step: float, world: int,
                   device) -> tuple:
    """Whole-job throughput of weak-scaled replicas: every rank processes
    `steps` x `units_per_step` units; the job takes as long as its slowest
    rank.  Returns (units per second over all ranks, max-over-ranks ms)."""
    total_ms = reduce_max(local_total_ms, world, device)
    return world * steps * units_per_step / (total_ms * 1e-3), total_ms


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# Rotation / rounding of the measured step (set from the command line in main).
ROT_NAMES = {"none": 0, "hadamard_det": 1, "hadamard_rand": 2}
ROUND_NAMES = {"rne": 0, "sr": 1}
MODE = {"rot": "hadamard_det", "rot_block": 32, "round": "rne", "seed": 0}


def mode_args():
    """(rot, rot_block, rnd, seed) as the C ABI and the oracle take them."""
    return (ROT_NAMES[MODE["rot"]], MODE["rot_block"], ROUND_NAMES[MODE["round"]], MODE["seed"])


def mode_text():
    rot = {"none": "no rotation", "hadamard_det": f"deterministic Hadamard {MODE['rot_block']}",
           "hadamard_rand": f"random-sign Hadamard {MODE['rot_block']}"}[MODE["rot"]]
    return f"{rot} along T, {MODE['round'].upper()}, seed {MODE['seed']}"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_sample(d, T, N, K, s_lines, seed=0, cores=1):
    """One bounded oracle sample: encode s_lines lines of each operand over the
    full T and contract them (s_lines^2 outputs).  With cores > 1 the oracle's
    calls are partitioned over threads (its C code releases the GIL): the
    encode by lines, the double GEMM by output rows; the arithmetic is the
    oracle's own.  Returns (seconds, flops)."""
    import numpy as np
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    rng = np.random.default_rng(seed)
    la = np.sort(rng.choice(N, s_lines, replace=False))
    lb = np.sort(rng.choice(K, s_lines, replace=False))
    rot, nb, rnd, qseed = mode_args()
    parts = max(1, min(cores, s_lines))
    t0 = time.perf_counter()
    with ThreadPoolExecutor(parts) as ex:
        qa = list(ex.map(lambda ln: oracle.quantize(d["dY"], oracle.CONTRACT_ROWS, rot, nb, rnd,
                                                    qseed, 1, lines=ln),
                         np.array_split(la, parts)))
        qb = list(ex.map(lambda ln: oracle.quantize(d["X"], oracle.CONTRACT_ROWS, rot, nb, rnd,
                                                    qseed, 2, lines=ln),
                         np.array_split(lb, parts)))
        Aq, As = np.concatenate([a[0] for a in qa]), np.concatenate([a[1] for a in qa])
        Bq, Bs = np.concatenate([b[0] for b in qb]), np.concatenate([b[1] for b in qb])
        edges = np.linspace(0, s_lines, parts + 1).astype(int)
        list(ex.map(lambda i: oracle.gemm_rows(Aq, As, Bq, Bs, int(edges[i]), int(edges[i + 1])),
                    range(parts)))
    return time.perf_counter() - t0, 2.0 * s_lines * s_lines * T


def calibrate_sample(d, T, N, K, budget_s, cores=1):
    """Lines per operand so that one oracle sample takes about budget_s
    (the contraction, quadratic in the lines, dominates the cost)."""
    dt, _ = oracle_sample(d, T, N, K, 64, cores=cores)
    s = int(64 * (budget_s / max(dt, 1e-6)) ** 0.5) // 16 * 16
    return max(16, min(s, N, K))


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    from workloads import config_inputs
    cfg, T, N, K = WORKLOADS[args.workload]
    d = config_inputs(cfg, seed=0, only=("dY", "X"))
    total_budget = args.ref_budget_s
    per_step = max(0.01, total_budget / max(1, args.steps + args.warmup))
    cores = host_cores()
    s = calibrate_sample(d, T, N, K, per_step, cores)
    for i in range(args.warmup):
        oracle_sample(d, T, N, K, s, seed=100 + i, cores=cores)
    times, flops = [], 0.0
    for i in range(args.steps):
        dt, f = oracle_sample(d, T, N, K, s, seed=i, cores=cores)
        times.append(dt)
        flops += f
    tot = sum(times)
    value = flops / tot / 1e12
    sample = (f"per step: {s} lines of dY and {s} lines of X (full T={T}) encoded with "
              f"{mode_text()}, then their {s}x{s} block of dW contracted in double; the "
              f"oracle's calls partitioned over {cores} host threads (encode by lines, "
              f"GEMM by output rows)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic",
            "config": workload_config(args, T, N, K),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(args, T, N, K):
    return {"workload": f"{args.workload} Wgrad: dY [{T},{N}] x X [{T},{K}] -> dW [{N},{K}] fp32, "
                        f"{mode_text()}, MXFP4 block 32",
            "T": T, "N": N, "K": K, "rot": MODE["rot"], "rot_block": MODE["rot_block"],
            "round": MODE["round"], "seed": MODE["seed"],
            "l2": "flushed before every timed step (512 MB write, outside the events)",
            "parallelism": "replicas" if args.gpus > 1 else "single-gpu"}


def run_mine(args, world, rank, local):
    import numpy as np
    import torch

    import mxfp4_precision_gb300 as mx
    from workloads import config_inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    cfg, T, N, K = WORKLOADS[args.workload]
    d = config_inputs(cfg, seed=0, only=("dY", "X"))
    dY_h = torch.from_numpy(d["dY"].view(np.int16)).pin_memory()
    X_h = torch.from_numpy(d["X"].view(np.int16)).pin_memory()
    dY = dY_h.to(dev)
    X = X_h.to(dev)
    stream = torch.cuda.current_stream(dev)
    L = mx.lib()
    sp = stream.cuda_stream
    rot, nb, rnd, seed = mode_args()

    aq = torch.empty(mx.codes_bytes(N, T), dtype=torch.uint8, device=dev)
    as_ = torch.empty(mx.scales_bytes(N, T), dtype=torch.uint8, device=dev)
    bq = torch.empty(mx.codes_bytes(K, T), dtype=torch.uint8, device=dev)
    bs = torch.empty(mx.scales_bytes(K, T), dtype=torch.uint8, device=dev)
    dW = torch.empty((N, K), dtype=torch.float32, device=dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    ptr = lambda t: t.data_ptr()

    # One step = the public Wgrad call on resident inputs: the encode of both
    # operands (one launch) and the GEMM.
    ws_step = torch.empty(mx.linear_workspace_bytes(mx.OP_WGRAD, T, N, K), dtype=torch.uint8,
                          device=dev)

    def step_call():
        yield L.mx_linear_wgrad(ptr(dY), ptr(X), ptr(dW), T, N, K, rot, nb, rnd, seed,
                                ptr(ws_step), ws_step.numel(), sp)

    # The two stand-alone launches, timed separately for the per-kernel rooflines.
    def step_parts():
        s1 = L.mx_quantize_pair(ptr(dY), T, N, ptr(X), T, K, rot, nb, rnd, seed, ptr(aq), ptr(as_),
                                ptr(bq), ptr(bs), sp)
        yield s1
        s2 = L.mx_gemm(ptr(aq), ptr(as_), ptr(bq), ptr(bs), ptr(dW), N, K, T, sp)
        yield s2

    def check(st, what):
        if st != 0:
            raise RuntimeError(f"{what} failed: {mx.status_string(st)}")

    # warm-up
    for _ in range(args.warmup):
        flush.zero_()
        for st in step_call():
            check(st, "warm-up")
        for st in step_parts():
            check(st, "warm-up")
    torch.cuda.synchronize(dev)
    mx.check_status()

    # Timed region: K steps, one pair of events per step (the flush between
    # steps stays outside them).
    n = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        for i in range(n):
            flush.zero_()
            ev[i][0].record(stream)
            for st in step_call():
                check(st, "step")
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    mx.check_status()
    step_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(n)]
    flops_step = 2.0 * N * K * T
    flops_per_s, total_ms = job_throughput(sum(step_ms), n, flops_step, world, dev)
    value = flops_per_s / 1e12

    # The stand-alone encode and GEMM launches (per-kernel rooflines), in
    # separate steps with an event between the two launches.
    nb_steps = min(n, 200)
    evb = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nb_steps)]
    for i in range(nb_steps):
        flush.zero_()
        evb[i][0].record(stream)
        for j, st in enumerate(step_parts()):
            check(st, "step")
            evb[i][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    mx.check_status()
    qp = [evb[i][0].elapsed_time(evb[i][1]) for i in range(nb_steps)]
    gm = [evb[i][1].elapsed_time(evb[i][2]) for i in range(nb_steps)]

    # ---- e2e: public call with host buffers, copies inside the timed region.
    # Every step copies its inputs host -> device, calls mx_linear_wgrad and
    # copies dW device -> host.  Steps are pipelined over three streams (input
    # copies, compute, output copies) with two device buffer sets, so step i+1's
    # input copy and step i-1's output copy overlap step i's compute, as in a
    # training loop that streams its layers.  The serial time (one step at a
    # time on one stream) is reported beside it.
    if not args.no_e2e:
        ws = torch.empty(mx.linear_workspace_bytes(mx.OP_WGRAD, T, N, K), dtype=torch.uint8,
                         device=dev)
        dW_h = [torch.empty((N, K), dtype=torch.float32).pin_memory() for _ in range(2)]
        dY_d = [torch.empty_like(dY) for _ in range(2)]
        X_d = [torch.empty_like(X) for _ in range(2)]
        dW_d = [dW, torch.empty_like(dW)]
    n_e2e = max(3, min(n, args.e2e_steps))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_cmp = stream

    def e2e_run(steps, pipelined):
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_cmp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        t0.record(s_in if pipelined else s_cmp)
        for i in range(steps):
            b = i % 2 if pipelined else 0
            if not pipelined:
                dY_d[b].copy_(dY_h, non_blocking=True)
                X_d[b].copy_(X_h, non_blocking=True)
                check(L.mx_linear_wgrad(ptr(dY_d[b]), ptr(X_d[b]), ptr(dW_d[b]), T, N, K, rot, nb,
                                        rnd, seed, ptr(ws), ws.numel(), sp), "e2e")
                dW_h[b].copy_(dW_d[b], non_blocking=True)
                continue
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_cmp[b])      # compute of step i-2 has read buffer b
                dY_d[b].copy_(dY_h, non_blocking=True)
                X_d[b].copy_(X_h, non_blocking=True)
                ev_in[b].record(s_in)
            s_cmp.wait_event(ev_in[b])
            if i >= 2:
                s_cmp.wait_event(ev_out[b])         # step i-2's dW[b] has been copied out
            check(L.mx_linear_wgrad(ptr(dY_d[b]), ptr(X_d[b]), ptr(dW_d[b]), T, N, K, rot, nb,
                                    rnd, seed, ptr(ws), ws.numel(), sp), "e2e")
            ev_cmp[b].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[b])
                dW_h[b].copy_(dW_d[b], non_blocking=True)
                ev_out[b].record(s_out)
        if pipelined:
            s_in.wait_stream(s_cmp)
            s_in.wait_stream(s_out)
        t1.record(s_in if pipelined else s_cmp)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1)

    e2e_value = e2e_ms = serial_ms = link = None
    if not args.no_e2e:
        e2e_run(2, True)                                 # warm-up
        e2e_ms = reduce_max(e2e_run(n_e2e, True), world, dev)
        serial_ms = e2e_run(n_e2e, False)
        mx.check_status()
        e2e_value = world * n_e2e * flops_step / (e2e_ms * 1e-3) / 1e12
        link = measure_link(dY_h, X_h, dW_h, dY_d, X_d, dW_d, s_in, s_out, dev)
        link["e2e_frac_of_both"] = ((dY_h.numel() * 2 + X_h.numel() * 2 + dW_h[0].numel() * 4)
                                    / (e2e_ms / n_e2e * 1e-3) / 1e9) / link["both_gbs"]

    # side measurement: the dual-output encode of dY (both backward encodings
    # from one read) against the two single-direction encodes it replaces
    dual = None
    if rank == 0 and not args.no_extras:
        dual = measure_dual(L, mx, dY, T, N, flush, stream, dev, hbm_gbs=load_peaks()[0]["hbm_gbs"])

    # the tensor cores' own MXFP4 rate on this GPU (issue-rate microbenchmark)
    # and the o_proj shape beside the headline workload
    fp4_meas = measure_fp4_peak(mx) if rank == 0 else None
    fused_side = None
    if rank == 0 and not args.no_extras:
        fused_side = measure_fused(L, mx, dY, X, dW, T, N, K, flush, stream, dev, step_ms,
                                   fp4_meas)
    fp8_side = nv_side = None
    peaks_var = None
    if rank == 0 and not args.no_extras:
        peaks_var = {"mxfp8": measure_mma_peak(mx, 5), "nvfp4": measure_mma_peak(mx, 2)}
        med = sorted(step_ms)[len(step_ms) // 2]
        fp8_side = measure_variant(L, mx, "mxfp8", dY, X, T, N, K, flush, stream, dev,
                                   peaks_var["mxfp8"], med)
        nv_side = measure_variant(L, mx, "nvfp4", dY, X, T, N, K, flush, stream, dev,
                                  peaks_var["nvfp4"], med)
    side = None
    if rank == 0 and not args.no_extras and args.workload != "o_proj":
        side = measure_side_workload(L, mx, "o_proj", dev, stream, flush, min(n, 300),
                                     args.warmup, fp4_meas, peaks_var)

    # parity spot check of the timed output (oracle entries, rank 0 only)
    parity = None
    if rank == 0 and not args.no_parity_check:
        parity = spot_check(d, dW, T, N, K)

    if rank != 0:
        return 0
    peaks, peak_src = load_peaks()
    fp4_peak = peaks["bf16_tflops"] * NOMINAL_FP4_OVER_BF16
    hbm = peaks["hbm_gbs"]
    q_bytes_n = N * T * (2 + 0.5 + 1 / 32)      # bf16 in, codes + scales out
    q_bytes_k = K * T * (2 + 0.5 + 1 / 32)
    mean = lambda v: sum(v) / len(v)
    t_q, t_g = mean(qp), mean(gm)
    traffic = load_traffic()
    wl = args.workload

    def tr(kernel, file):
        # The captures are of the default mode (deterministic Hadamard 32,
        # round to nearest); another mode runs other kernel code.
        if (MODE["rot"], MODE["rot_block"], MODE["round"]) != ("hadamard_det", 32, "rne"):
            return None
        hit = traffic.get((kernel, wl))
        if hit and hit[0] == kernel_source_hash(file):
            return hit[1]
        return None

    g_ach = flops_step / (t_g * 1e-3) / 1e12
    gemm_rf = {"kernel": "mx_gemm_kernel", "bound": "tensor",
               "achieved": g_ach,
               "peak": fp4_peak, "unit": "TFLOP/s",
               "frac": g_ach / fp4_peak,
               "traffic": tr("mx_gemm_kernel", "mx_gemm.cu"),
               "peak_basis": f"{peak_src} bf16 burst {peaks['bf16_tflops']} TFLOP/s x nominal "
                             f"fp4/bf16 ratio {NOMINAL_FP4_OVER_BF16:g}",
               "peak_fp4_measured": fp4_meas["tflops"],
               "frac_fp4_measured": g_ach / fp4_meas["tflops"],
               "ms_per_launch": t_g}
    quant_rf = {"kernel": "mxq_colwise_kernel", "bound": "hbm",
                "achieved": (q_bytes_n + q_bytes_k) / (t_q * 1e-3) / 1e9,
                "peak": hbm, "unit": "GB/s",
                "frac": (q_bytes_n + q_bytes_k) / (t_q * 1e-3) / 1e9 / hbm,
                "traffic": tr("mxq_colwise_kernel", "mx_quant.cu"),
                "peak_basis": f"{peak_src} HBM copy bandwidth",
                "ms_per_launch": t_q}
    kernels = [gemm_rf, quant_rf]
    dominant = gemm_rf if t_g >= t_q else quant_rf
    clk = clocks.summary()
    cpu = None
    if not args.no_cpu_baseline:
        cores = host_cores()
        s = calibrate_sample(d, T, N, K, args.cpu_budget_s, cores)
        dt, f = oracle_sample(d, T, N, K, s, cores=cores)
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{s} lines of dY and {s} lines of X (full T={T}) encoded "
                         f"({mode_text()}), then their {s}x{s} block of dW contracted "
                         f"in double; the oracle's calls partitioned over {cores} host "
                         f"threads (encode by lines, GEMM by output rows); {dt:.1f} s"}
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": n, "warmup": args.warmup, "ms_per_step": total_ms / n,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "mxfp4 (e2m1 x e8m0, fp32 accumulate)", "data": "synthetic",
            "config": workload_config(args, T, N, K),
            "roofline": {k: dominant[k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                                   "traffic", "peak_fp4_measured",
                                                   "frac_fp4_measured") if k in dominant},
            "roofline_kernels": kernels,
            "step_launches": 2,
            "fused_wgrad": fused_side,
            "fp8_comparator": fp8_side,
            "nvfp4_variant": nv_side,
            "fp4_peak_fraction": value / fp4_peak,
            "fp4_peak_measured": fp4_meas,
            "fp4_measured_fraction": value / fp4_meas["tflops"],
            "o_proj": side,
            "breakdown_ms": {"quantize_pair": t_q, "gemm": t_g,
                             "note": f"the stand-alone encode and GEMM launches, in separate "
                                     f"{nb_steps} steps with an event between them (the "
                                     f"headline step is mx_linear_wgrad: the same two launches)"},
            "cpu_baseline": cpu,
            "e2e": None if e2e_ms is None else {
                "value": e2e_value, "unit": "TFLOP/s",
                "h2d_bytes_per_step": dY_h.numel() * 2 + X_h.numel() * 2,
                "d2h_bytes_per_step": dW_h[0].numel() * 4,
                "ms_per_step": e2e_ms / n_e2e, "call": "mx_linear_wgrad",
                "schedule": "steps pipelined over input-copy / compute / output-copy "
                            "streams, two device buffer sets",
                "serial_ms_per_step": serial_ms / n_e2e,
                "serial_value": world * n_e2e * flops_step / (serial_ms * 1e-3) / 1e12,
                "host_link": link},
            "gpu_launches": 2 * n,
            "dual_quantiser": dual,
            "clocks": clk,
            "parity_spot_check": parity}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def measure_fp4_peak(mx, reps=3):
    """All-SM issue rate of the GEMM's own instruction,
    tcgen05.mma.cta_group::2.kind::mxf4.block_scale (M=256, N=256, K=64), on
    operands resident in shared memory (mx_bench_mma); best of `reps`."""
    best = None
    for _ in range(reps):
        r = mx.bench_mma(kind=0, cta_group=2, n=256, mmas_per_iter=4, iters=20000)
        if best is None or r["tflops"] > best["tflops"]:
            best = r
    return {"tflops": best["tflops"], "ns_per_mma": best["ns_per_mma"], "ctas": best["ctas"],
            "instruction": "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X "
                           "M=256 N=256 K=64, operands in shared memory, no copies",
            "call": "mx_bench_mma", "best_of": reps}


def measure_side_workload(L, mx, name, dev, stream, flush, steps, warmup, fp4_meas,
                          peaks_var=None):
    """Quantise-pair + GEMM of another Wgrad shape, timed like the headline
    (L2 flushed before every step, CUDA events on the launching stream)."""
    import numpy as np
    import torch
    from workloads import config_inputs
    cfg, T, N, K = WORKLOADS[name]
    d = config_inputs(cfg, seed=0, only=("dY", "X"))
    dY = torch.from_numpy(d["dY"].view(np.int16)).to(dev)
    X = torch.from_numpy(d["X"].view(np.int16)).to(dev)
    sp = stream.cuda_stream
    rot, nb, rnd, seed = mode_args()
    aq = torch.empty(mx.codes_bytes(N, T), dtype=torch.uint8, device=dev)
    as_ = torch.empty(mx.scales_bytes(N, T), dtype=torch.uint8, device=dev)
    bq = torch.empty(mx.codes_bytes(K, T), dtype=torch.uint8, device=dev)
    bs = torch.empty(mx.scales_bytes(K, T), dtype=torch.uint8, device=dev)
    dW = torch.empty((N, K), dtype=torch.float32, device=dev)
    ptr = lambda t: t.data_ptr()

    def parts():
        yield L.mx_quantize_pair(ptr(dY), T, N, ptr(X), T, K, rot, nb, rnd, seed, ptr(aq),
                                 ptr(as_), ptr(bq), ptr(bs), sp)
        yield L.mx_gemm(ptr(aq), ptr(as_), ptr(bq), ptr(bs), ptr(dW), N, K, T, sp)

    for _ in range(warmup):
        flush.zero_()
        if any(parts()):
            raise RuntimeError(f"{name}: launch failed")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    whole = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    torch.cuda.synchronize(dev)
    ws = torch.empty(mx.linear_workspace_bytes(mx.OP_WGRAD, T, N, K), dtype=torch.uint8, device=dev)

    def call():
        return L.mx_linear_wgrad(ptr(dY), ptr(X), ptr(dW), T, N, K, rot, nb, rnd, seed, ptr(ws),
                                 ws.numel(), sp)

    for _ in range(warmup):
        flush.zero_()
        if call():
            raise RuntimeError(f"{name}: launch failed")
    for i in range(steps):
        flush.zero_()
        whole[i][0].record(stream)
        if call():
            raise RuntimeError(f"{name}: launch failed")
        whole[i][1].record(stream)
    for i in range(steps):
        flush.zero_()
        ev[i][0].record(stream)
        for j, st in enumerate(parts()):
            if st != 0:
                raise RuntimeError(f"{name}: launch failed")
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    mx.check_status()
    t_step = sum(whole[i][0].elapsed_time(whole[i][1]) for i in range(steps)) / steps
    t_q = sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(steps)) / steps
    t_g = sum(ev[i][1].elapsed_time(ev[i][2]) for i in range(steps)) / steps
    flops = 2.0 * N * K * T
    hbm = load_peaks()[0]["hbm_gbs"]
    qbytes = (N + K) * T * (2 + 0.5 + 1 / 32)
    fp8 = nv = None
    if peaks_var is not None:
        fp8 = measure_variant(L, mx, "mxfp8", dY, X, T, N, K, flush, stream, dev,
                              peaks_var["mxfp8"], t_step)
        nv = measure_variant(L, mx, "nvfp4", dY, X, T, N, K, flush, stream, dev,
                             peaks_var["nvfp4"], t_step)
    return {"workload": f"{name} Wgrad: dY [{T},{N}] x X [{T},{K}] -> dW [{N},{K}] fp32, "
                        f"{mode_text()}",
            "fp8_comparator": fp8, "nvfp4_variant": nv,
            "steps": steps, "ms_per_step": t_step,
            "value": flops / (t_step * 1e-3) / 1e12, "unit": "TFLOP/s",
            "step_launches": 2,
            "breakdown_ms": {"quantize_pair": t_q, "gemm": t_g},
            "gemm_tflops": flops / (t_g * 1e-3) / 1e12,
            "gemm_frac_fp4_measured": flops / (t_g * 1e-3) / 1e12 / fp4_meas["tflops"],
            "quantizer_gbs": qbytes / (t_q * 1e-3) / 1e9,
            "quantizer_frac_hbm": qbytes / (t_q * 1e-3) / 1e9 / hbm}


def measure_fused(L, mx, dY, X, dW, T, N, K, flush, stream, dev, step_ms, fp4_meas, reps=50):
    """mx_linear_wgrad_fused (the encode inside the GEMM's launch) on the
    headline workload: time per call (L2 flushed before each) beside the
    two-launch step, and whether its output has the same bits."""
    import torch
    rot, nb, rnd, seed = mode_args()
    if not L.mx_linear_wgrad_fused_supported(T, N, K, rot, nb, rnd):
        return {"call": "mx_linear_wgrad_fused", "supported": False}
    sp = stream.cuda_stream
    ptr = lambda t: t.data_ptr()
    ws = torch.empty(mx.linear_workspace_bytes(mx.OP_WGRAD, T, N, K), dtype=torch.uint8, device=dev)
    out = torch.empty_like(dW)

    def call():
        st = L.mx_linear_wgrad_fused(ptr(dY), ptr(X), ptr(out), T, N, K, rot, nb, rnd, seed,
                                     ptr(ws), ws.numel(), sp)
        if st != 0:
            raise RuntimeError(f"mx_linear_wgrad_fused: {mx.status_string(st)}")
    for _ in range(3):
        flush.zero_()
        call()
    ts = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ts.append(e0.elapsed_time(e1))
    mx.check_status()
    t = sorted(ts)[len(ts) // 2]
    same = bool(torch.equal(out.view(torch.int32), dW.view(torch.int32)))
    two = sorted(step_ms)[len(step_ms) // 2]
    return {"call": "mx_linear_wgrad_fused", "supported": True, "ms": t, "median_of": reps,
            "tflops": 2.0 * N * K * T / (t * 1e-3) / 1e12,
            "two_launch_step_ms_median": two,
            "bitwise_equal_to_two_launch_step": same}


def measure_mma_peak(mx, kind, reps=3):
    """All-SM issue rate of a variant GEMM's instruction (mx_bench_mma, pair
    form, M=256 N=256, operands in shared memory); best of `reps`.  kind 5:
    kind::mxf8f6f4 scale_vec::1X (MXFP8, K=32); kind 2: kind::mxf4nvf4
    scale_vec::4X (NVFP4, K=64)."""
    best = None
    for _ in range(reps):
        r = mx.bench_mma(kind=kind, cta_group=2, n=256, mmas_per_iter=4, iters=20000)
        if best is None or r["tflops"] > best["tflops"]:
            best = r
    name = {5: "kind::mxf8f6f4.block_scale.scale_vec::1X M=256 N=256 K=32",
            2: "kind::mxf4nvf4.block_scale.scale_vec::4X M=256 N=256 K=64"}[kind]
    return {"tflops": best["tflops"], "ns_per_mma": best["ns_per_mma"],
            "instruction": "tcgen05.mma.cta_group::2." + name, "call": "mx_bench_mma",
            "best_of": reps}


def measure_variant(L, mx, fmt, dY, X, T, N, K, flush, stream, dev, peak, mxfp4_step_ms,
                    reps=50):
    """Another element format on the same Wgrad shape, through its public
    call: "mxfp8" (the FP8 comparator: MXFP8 encode of both operands + the
    MXFP8 GEMM, no rotation) or "nvfp4" (the NVFP4 variant: tensor-amax and
    encode launches + the NVFP4 GEMM, deterministic Hadamard 16), and its GEMM
    launch alone; medians over `reps` calls, L2 flushed before each."""
    import torch
    sp = stream.cuda_stream
    ptr = lambda t: t.data_ptr()
    nv = fmt == "nvfp4"
    wsb = (mx.linear_wgrad_nvfp4_workspace_bytes(T, N, K) if nv
           else mx.linear_wgrad_mxfp8_workspace_bytes(T, N, K))
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    out = torch.empty((N, K), dtype=torch.float32, device=dev)
    align = lambda x: (x + 255) // 256 * 256
    codes = mx.codes_bytes if nv else mx.mxfp8_codes_bytes
    scales = mx.nvfp4_scales_bytes if nv else mx.scales_bytes
    o_as = align(codes(N, T))
    o_bq = o_as + align(scales(N, T))
    o_bs = o_bq + align(codes(K, T))
    o_am = o_bs + align(scales(K, T))
    base = ws.data_ptr()

    def step():
        if nv:
            return L.mx_linear_wgrad_nvfp4(ptr(dY), ptr(X), ptr(out), T, N, K,
                                           mx.ROT_HADAMARD_DET, 16, 0, base, ws.numel(), sp)
        return L.mx_linear_wgrad_mxfp8(ptr(dY), ptr(X), ptr(out), T, N, K, base, ws.numel(), sp)

    def gemm():
        if nv:
            return L.mx_gemm_nvfp4(base, base + o_as, base + o_am, base + o_bq, base + o_bs,
                                   base + o_am + 4, ptr(out), N, K, T, sp)
        return L.mx_gemm_mxfp8(base, base + o_as, base + o_bq, base + o_bs, ptr(out), N, K, T, sp)

    def timed(fn):
        for _ in range(3):
            flush.zero_()
            if fn():
                raise RuntimeError("MXFP8 comparator launch failed")
        ts = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1))
        return sorted(ts)[len(ts) // 2]

    t_step = timed(step)
    t_gemm = timed(gemm)             # on the operands the last step left in the workspace
    mx.check_status()
    flops = 2.0 * N * K * T
    return {"call": "mx_linear_wgrad_nvfp4" if nv else "mx_linear_wgrad_mxfp8",
            "format": ("NVFP4: E2M1 in blocks of 16 along T, UE4M3 block scale, fp32 tensor "
                       "scale, deterministic Hadamard 16, round to nearest even") if nv else
                      ("MXFP8: E4M3 elements, E8M0 scale per 32 along T, no rotation, round "
                       "to nearest even"),
            "ms_per_step": t_step, "tflops": flops / (t_step * 1e-3) / 1e12,
            "gemm_ms": t_gemm, "gemm_tflops": flops / (t_gemm * 1e-3) / 1e12,
            "peak_measured": peak,
            "gemm_frac_peak_measured": flops / (t_gemm * 1e-3) / 1e12 / peak["tflops"],
            "mxfp4_step_speedup": t_step / mxfp4_step_ms, "median_of": reps,
            "step_launches": 3 if nv else 2}


def measure_link(dY_h, X_h, dW_h, dY_d, X_d, dW_d, s_in, s_out, dev, reps=5):
    """The host link on its own, for the e2e figure's roofline: the step's input copies host -> device
    alone, its dW copy device -> host alone, and both at once on the two copy streams (median of
    ``reps``).  ``e2e_frac_of_both`` is then the e2e step's bytes per second over the both-ways rate."""
    import torch
    def run(fn):
        ts = []
        for r in range(reps + 1):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            cur = torch.cuda.current_stream(dev)
            a.record(cur)
            s_in.wait_stream(cur)
            s_out.wait_stream(cur)
            fn()
            cur.wait_stream(s_in)
            cur.wait_stream(s_out)
            b.record(cur)
            torch.cuda.synchronize(dev)
            if r:
                ts.append(a.elapsed_time(b))
        ts.sort()
        return ts[len(ts) // 2]

    def h2d():
        with torch.cuda.stream(s_in):
            dY_d[1].copy_(dY_h, non_blocking=True)
            X_d[1].copy_(X_h, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s_out):
            dW_h[1].copy_(dW_d[1], non_blocking=True)

    def both():
        h2d()
        d2h()

    bi, bo = dY_h.numel() * 2 + X_h.numel() * 2, dW_h[1].numel() * 4
    t_in, t_out, t_both = run(h2d), run(d2h), run(both)
    return {"h2d_gbs": bi / (t_in * 1e-3) / 1e9, "d2h_gbs": bo / (t_out * 1e-3) / 1e9,
            "both_gbs": (bi + bo) / (t_both * 1e-3) / 1e9,
            "note": "plain copies of the step's own buffers on the e2e copy streams; the link is "
                    "the e2e bound (both directions share it)"}


def measure_dual(L, mx, dY, T, N, flush, stream, dev, hbm_gbs, reps=30):
    """mx_quantize_dual on dY [T, N] vs mx_quantize along T (rotated) + along N,
    each rep after an L2 flush; algorithmic bytes 2 (bf16 read) + 2 x 0.53125."""
    import torch
    sp = stream.cuda_stream
    ptr = lambda t: t.data_ptr()
    ct = torch.empty(mx.codes_bytes(N, T), dtype=torch.uint8, device=dev)
    st = torch.empty(mx.scales_bytes(N, T), dtype=torch.uint8, device=dev)
    cn = torch.empty(mx.codes_bytes(T, N), dtype=torch.uint8, device=dev)
    sn = torch.empty(mx.scales_bytes(T, N), dtype=torch.uint8, device=dev)
    rot, nb = mx.ROT_HADAMARD_DET, 32

    def dual():
        return [L.mx_quantize_dual(ptr(dY), T, N, rot, nb, 0, 0, ptr(ct), ptr(st), ptr(cn),
                                   ptr(sn), sp)]

    def separate():
        return [L.mx_quantize(ptr(dY), T, N, mx.CONTRACT_ROWS, rot, nb, 0, 0, ptr(ct), ptr(st), sp),
                L.mx_quantize(ptr(dY), T, N, mx.CONTRACT_COLS, mx.ROT_NONE, 32, 0, 0, ptr(cn),
                              ptr(sn), sp)]

    def timed(fn):
        for _ in range(3):
            flush.zero_()
            if any(fn()):
                raise RuntimeError("dual-output measurement launch failed")
        ts = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1))
        return sorted(ts)[len(ts) // 2]

    t_dual, t_sep = timed(dual), timed(separate)
    mx.check_status()
    nbytes = T * N * (2 + 2 * (0.5 + 1 / 32))
    return {"call": "mx_quantize_dual", "input": f"dY [{T},{N}] bf16",
            "outputs": "along T (det-Hadamard 32, Wgrad operand) + along N (no rotation, "
                       "Dgrad operand), RNE",
            "ms": t_dual, "ms_two_separate_launches": t_sep,
            "achieved_gbs": nbytes / (t_dual * 1e-3) / 1e9, "peak_gbs": hbm_gbs,
            "frac": nbytes / (t_dual * 1e-3) / 1e9 / hbm_gbs,
            "algorithmic_bytes": nbytes, "median_of": reps}


def run_sweep(args):
    """The measurements beside the headline (one GPU, one JSON line each):
    the rotation / rounding ablation at down_proj shapes with its quantisation
    error, the down_proj Hadamard-size sweep, the six GEMMs of the QKV +
    gate/up layers, and a cuBLAS bf16 GEMM of the Wgrad shapes for context."""
    import numpy as np
    import torch

    import mxfp4_precision_gb300 as mx
    import oracle
    from workloads import bf16_bits_to_f32, config_inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    L = mx.lib()
    ptr = lambda t: t.data_ptr()
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    peaks, _ = load_peaks()
    fp4_peak = peaks["bf16_tflops"] * NOMINAL_FP4_OVER_BF16
    fp4_meas = measure_fp4_peak(mx)["tflops"]
    reps = args.sweep_reps

    def timed(fn):
        for _ in range(2):
            flush.zero_()
            fn()
        ts = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1))
        mx.check_status()
        return sorted(ts)[len(ts) // 2]

    def ok(st, what):
        if st != 0:
            raise RuntimeError(f"{what}: {mx.status_string(st)}")

    def emit(obj):
        print(json.dumps(obj), flush=True)

    # ---- down_proj shapes: ablation modes and Hadamard sizes
    T, N, K = 8192, 4096, 14336
    d = config_inputs("down_proj", seed=0, only=("dY", "X"))
    dY = torch.from_numpy(d["dY"].view(np.int16)).to(dev)
    X = torch.from_numpy(d["X"].view(np.int16)).to(dev)
    aq = torch.empty(mx.codes_bytes(N, T), dtype=torch.uint8, device=dev)
    as_ = torch.empty(mx.scales_bytes(N, T), dtype=torch.uint8, device=dev)
    bq = torch.empty(mx.codes_bytes(K, T), dtype=torch.uint8, device=dev)
    bs = torch.empty(mx.scales_bytes(K, T), dtype=torch.uint8, device=dev)
    dW = torch.empty((N, K), dtype=torch.float32, device=dev)
    flops = 2.0 * N * K * T
    qbytes = (N + K) * T * (2 + 0.5 + 1 / 32)

    def quant(rot, nb, rnd, seed):
        ok(L.mx_quantize_pair(ptr(dY), T, N, ptr(X), T, K, rot, nb, rnd, seed, ptr(aq), ptr(as_),
                              ptr(bq), ptr(bs), sp), "quantize_pair")

    def gemm():
        ok(L.mx_gemm(ptr(aq), ptr(as_), ptr(bq), ptr(bs), ptr(dW), N, K, T, sp), "gemm")

    rng = np.random.default_rng(7)
    la = np.sort(rng.choice(N, 32, replace=False))
    lb = np.sort(rng.choice(K, 32, replace=False))
    rows = np.sort(rng.choice(N, 16, replace=False))
    dyf = bf16_bits_to_f32(d["dY"]).astype(np.float64)
    xf = bf16_bits_to_f32(d["X"]).astype(np.float64)
    exact = dyf[:, rows].T @ xf                     # rows of dY^T X, in double

    def element_rms(bits, lines, rot, nb, rnd, seed, tag):
        codes, scales = oracle.quantize(bits, oracle.CONTRACT_ROWS, rot, nb, rnd, seed, tag,
                                        lines=lines)
        deq = oracle.dequantize(codes, scales)
        r = np.stack([oracle.rotate_line(bits[:, c], rot, nb, seed) for c in lines]).astype(
            np.float64)
        return float(np.sqrt(((deq - r) ** 2).sum() / (r ** 2).sum()))

    for name, rot, nb, rnd, seed in [("none", mx.ROT_NONE, 32, mx.ROUND_RNE, 0),
                                     ("hadamard_det_32", mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE, 0),
                                     ("hadamard_rand_32", mx.ROT_HADAMARD_RAND, 32, mx.ROUND_RNE, 1),
                                     ("sr", mx.ROT_NONE, 32, mx.ROUND_SR, 1)]:
        t_q = timed(lambda: quant(rot, nb, rnd, seed))
        quant(rot, nb, rnd, seed)
        t_g = timed(gemm)
        got = dW[torch.from_numpy(rows).to(dev)].double().cpu().numpy()
        out_rms = float(np.linalg.norm(got - exact) / np.linalg.norm(exact))
        emit({"sweep": "ablation", "workload": f"down_proj Wgrad T={T} N={N} K={K}", "mode": name,
              "quantize_pair_ms": t_q, "gemm_ms": t_g,
              "tflops_incl_quant": flops / ((t_q + t_g) * 1e-3) / 1e12,
              "quantizer_gbs": qbytes / (t_q * 1e-3) / 1e9,
              "element_rel_rms": {"dY": element_rms(d["dY"], la, rot, nb, rnd, seed, 1),
                                  "X": element_rms(d["X"], lb, rot, nb, rnd, seed, 2),
                                  "sample": "32 channels of each operand, full T, rotated domain"},
              "output_rel_rms": out_rms,
              "output_sample": "16 rows of dW (all 14336 columns) against dY^T X in double",
              "graded": False})

    for nb in (16, 32, 64, 128, 256):
        t_q = timed(lambda: quant(mx.ROT_HADAMARD_DET, nb, mx.ROUND_RNE, 0))
        quant(mx.ROT_HADAMARD_DET, nb, mx.ROUND_RNE, 0)
        t_g = timed(gemm)
        emit({"sweep": "hadamard_size", "workload": f"down_proj Wgrad T={T} N={N} K={K}",
              "rot_block": nb, "quantize_pair_ms": t_q, "gemm_ms": t_g,
              "quantizer_gbs": qbytes / (t_q * 1e-3) / 1e9,
              "quantizer_frac_hbm": qbytes / (t_q * 1e-3) / 1e9 / peaks["hbm_gbs"],
              "gemm_tflops": flops / (t_g * 1e-3) / 1e12,
              "gemm_frac_fp4": flops / (t_g * 1e-3) / 1e12 / fp4_peak,
              "gemm_frac_fp4_measured": flops / (t_g * 1e-3) / 1e12 / fp4_meas,
              "tflops_incl_quant": flops / ((t_q + t_g) * 1e-3) / 1e12})

    # cuBLASLt's block-scaled FP4 GEMM on the same encoded operands (context only, not the
    # path; optional: reported as unavailable where this torch build does not take FP4)
    quant(mx.ROT_HADAMARD_DET, 32, mx.ROUND_RNE, 0)
    gemm()
    try:
        fa = aq.view(torch.float4_e2m1fn_x2).view(N, T // 2)
        fb = bq.view(torch.float4_e2m1fn_x2).view(K, T // 2)
        sa, sb = as_.view(torch.float8_e8m0fnu), bs.view(torch.float8_e8m0fnu)
        lib_mm = lambda: torch._scaled_mm(fa, fb.t(), sa, sb, out_dtype=torch.bfloat16)
        ref = lib_mm().float()
        torch.cuda.synchronize(dev)
        rel = float((ref - dW).norm() / dW.norm())
        t_l = timed(lib_mm)
        emit({"sweep": "cublaslt_mxfp4_reference", "workload": f"down_proj Wgrad T={T} N={N} K={K}",
              "call": "torch._scaled_mm(float4_e2m1fn_x2, float8_e8m0fnu scales), bf16 out",
              "ms": t_l, "tflops": flops / (t_l * 1e-3) / 1e12,
              "rel_diff_vs_mx_gemm": rel,
              "note": "same codes and tiled scales as mx_gemm; its output rounds to bf16"})
    except Exception as e:                       # not offered by this torch / cuBLASLt
        emit({"sweep": "cublaslt_mxfp4_reference", "unavailable": f"{type(e).__name__}: {e}"[:300]})

    # cuBLAS bf16 GEMM of the same Wgrad shapes (context only, not the path)
    for wl, (tt, nn, kk) in (("o_proj", (8192, 4096, 4096)), ("down_proj", (T, N, K))):
        a = dY.view(torch.bfloat16)[:tt, :nn]
        b = X.view(torch.bfloat16)[:tt, :kk]
        t_b = timed(lambda: torch.matmul(a.t(), b))
        emit({"sweep": "cublas_bf16_reference", "workload": f"{wl} Wgrad shape T={tt} N={nn} K={kk}",
              "call": "torch.matmul(dY.t(), X), bf16 in and out", "ms": t_b,
              "tflops": 2.0 * nn * kk * tt / (t_b * 1e-3) / 1e12})
    del dY, X, aq, as_, bq, bs, dW, d
    torch.cuda.empty_cache()

    # ---- QKV + gate/up: Fprop, Dgrad and Wgrad of both weights (six GEMMs)
    T4 = 16384
    d4 = config_inputs("qkv_gateup", seed=0)
    t4 = {k: torch.from_numpy(v.view(np.int16)).to(dev) for k, v in d4.items()}
    del d4
    total_ms, total_flops = 0.0, 0.0
    for w, dy in (("W_qkv", "dY_qkv"), ("W_gu", "dY_gu")):
        Wt, dYt, Xt = t4[w], t4[dy], t4["X"]
        Nw, Kx = Wt.shape[0], Xt.shape[1]
        for op, fn, a, b, shape, rot in (
                ("fprop", "mx_linear_fprop", Xt, Wt, (T4, Nw), mx.ROT_NONE),
                ("dgrad", "mx_linear_dgrad", dYt, Wt, (T4, Kx), mx.ROT_NONE),
                ("wgrad", "mx_linear_wgrad", dYt, Xt, (Nw, Kx), mx.ROT_HADAMARD_DET)):
            opc = {"fprop": mx.OP_FPROP, "dgrad": mx.OP_DGRAD, "wgrad": mx.OP_WGRAD}[op]
            ws = torch.empty(max(256, mx.linear_workspace_bytes(opc, T4, Nw, Kx)),
                             dtype=torch.uint8, device=dev)
            out = torch.empty(shape, dtype=torch.float32, device=dev)
            f = getattr(L, fn)
            run = lambda: ok(f(ptr(a), ptr(b), ptr(out), T4, Nw, Kx, rot, 32, mx.ROUND_RNE, 0,
                               ptr(ws), ws.numel(), sp), fn)
            t_op = timed(run)
            fl = 2.0 * T4 * Nw * Kx
            total_ms += t_op
            total_flops += fl
            emit({"sweep": "qkv_gateup", "weight": w, "op": op, "call": fn,
                  "shape": {"T": T4, "N": Nw, "K": Kx}, "ms": t_op,
                  "tflops_incl_quant": fl / (t_op * 1e-3) / 1e12})
            del ws, out
    emit({"sweep": "qkv_gateup", "op": "all six", "ms": total_ms,
          "gflop": total_flops / 1e9, "tflops_incl_quant": total_flops / (total_ms * 1e-3) / 1e12})
    del t4
    torch.cuda.empty_cache()

    # ---- the oracle at full size on this host (a reported baseline, not the target):
    # its encode single-threaded, its double GEMM partitioned by output columns over
    # every host core (the oracle's C calls release the GIL; arithmetic unchanged)
    from concurrent.futures import ThreadPoolExecutor
    cores = host_cores()
    for name in ("tiny", "o_proj", "down_proj"):
        cfg, T_, N_, K_ = ("tiny", 256, 128, 256) if name == "tiny" else WORKLOADS[name]
        dd = config_inputs(cfg, seed=0, only=("dY", "X"))
        t0 = time.perf_counter()
        Aq, As = oracle.quantize(dd["dY"], oracle.CONTRACT_ROWS, oracle.ROT_HADAMARD_DET, 32,
                                 oracle.ROUND_RNE, 0, 1)
        Bq, Bs = oracle.quantize(dd["X"], oracle.CONTRACT_ROWS, oracle.ROT_HADAMARD_DET, 32,
                                 oracle.ROUND_RNE, 0, 2)
        tq = time.perf_counter() - t0
        edges = np.linspace(0, K_, max(1, min(cores, K_ // 8)) + 1).astype(int)
        t0 = time.perf_counter()
        with ThreadPoolExecutor(len(edges) - 1) as ex:
            list(ex.map(lambda i: oracle.gemm(Aq, As, Bq[edges[i]:edges[i + 1]],
                                              Bs[edges[i]:edges[i + 1]]), range(len(edges) - 1)))
        tg = time.perf_counter() - t0
        fl = 2.0 * N_ * K_ * T_
        emit({"sweep": "oracle_full_size", "workload": f"{name} Wgrad T={T_} N={N_} K={K_}, "
              "deterministic Hadamard 32, RNE", "encode_s_one_core": tq,
              "gemm_s": tg, "gemm_threads": len(edges) - 1, "host_cores": cores,
              "tflops_incl_encode": fl / (tq + tg) / 1e12})
        del dd, Aq, As, Bq, Bs
    return 0


def spot_check(d, dW, T, N, K):
    """Oracle check of 32 x 32 sampled entries of the timed dW."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(123)
    ia = np.sort(rng.choice(N, 32, replace=False))
    jb = np.sort(rng.choice(K, 32, replace=False))
    rot, nb, rnd, qseed = mode_args()
    Aq, As = oracle.quantize(d["dY"], oracle.CONTRACT_ROWS, rot, nb, rnd, qseed, 1, lines=ia)
    Bq, Bs = oracle.quantize(d["X"], oracle.CONTRACT_ROWS, rot, nb, rnd, qseed, 2, lines=jb)
    C, Ca = oracle.gemm(Aq, As, Bq, Bs)
    got = dW.cpu().numpy()[np.ix_(ia, jb)].astype(np.float64)
    ratio = float((np.abs(got - C) / np.maximum(Ca, 1e-300)).max())
    return {"entries": 1024, "max_err_over_sum_abs": ratio, "pass": ratio <= 1e-5}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["mine", "reference"], default="mine")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="down_proj")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget-s", type=float, default=8.0)
    ap.add_argument("--ref-budget-s", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-parity-check", action="store_true")
    ap.add_argument("--rot", choices=sorted(ROT_NAMES), default="hadamard_det",
                    help="rotation of both operands along T (default: deterministic Hadamard)")
    ap.add_argument("--rot-block", type=int, choices=[16, 32, 64, 128, 256], default=32)
    ap.add_argument("--round", choices=sorted(ROUND_NAMES), default="rne")
    ap.add_argument("--seed", type=int, default=0, help="sign / SR seed")
    ap.add_argument("--sweep", action="store_true",
                    help="print the ablation / Hadamard-size / QKV+gate-up / cuBLAS reference "
                         "measurements instead of the headline line (one GPU)")
    ap.add_argument("--sweep-reps", type=int, default=10)
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the side measurements (o_proj shape, dual-output encode)")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end host-buffer leg (for profiler captures of the "
                         "hot path only; the line then has no e2e number)")
    args = ap.parse_args()
    MODE.update(rot=args.rot, rot_block=args.rot_block, round=args.round, seed=args.seed)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    if args.sweep:
        return run_sweep(args) if rank == 0 else 0
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_mine(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
