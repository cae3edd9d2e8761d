#!/usr/bin/env python3
"""Benchmark of the fused decode-attention step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--cluster-size C] [--stages S]

Prints ONE JSON line (rank 0). A step is one fused decode step (QKV projection,
KV append, attention, output projection) of the workload over one batch; the
default workload is the Llama2-7B-shaped block at B=1, ctx_len 4096.

value    = achieved HBM GB/s over the step's algorithmic bytes (both weights +
           the K/V cache rows read), summed over ranks: total bytes / max
           over ranks of the timed region.
e2e      = the same metric through the host-buffer C-ABI entry point
           (cfa_decode_step_host): every step copies x host->device, runs the
           kernel, copies out device->host and synchronizes.
roofline = the fused kernel (the dominant kernel of a step) against the measured
           HBM copy bandwidth.
cpu_baseline / --impl reference = the fp64 CPU oracle on the host cores (cpu_baseline
           at N = 1 only: under torchrun the line carries none).

Inputs live in three rotating copies (each larger than the 129 MB L2), so no
step reads what the previous step left in L2. Multi-GPU runs are independent
replicas (the step has no exchange between GPUs).

--workload mla_v3_b1_ctx4k (or another MLA workload) measures a
DeepSeek-style latent-attention step (4 launches); its bytes are every weight
of the block plus the latent cache rows read.

--workload llama7b_32l_b1_ctx1k (or another layer stack) measures the decode
loop instead: a step is one token through every layer (RMSNorm, the fused
attention block, residual, RMSNorm + SwiGLU MLP, residual), replayed from one
CUDA graph; its bytes are all layers' weight matrices plus the cache rows
read (13.5 GB per token for 32 Llama2-7B layers, far above L2).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused decode-attn step latency (µs) and achieved HBM GB/s vs GB300 peak"
DEFAULT_WORKLOAD = "llama7b_b1_ctx4k"
FALLBACK_HBM_GBS = 6800.0
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASON_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


# ------------------------------------------------------------ host helpers


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cluster-size", type=int, default=None)
    ap.add_argument("--stages", type=int, default=None)
    ap.add_argument("--copies", type=int, default=3)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--preload-seconds", type=float, default=1.0,
                    help="untimed load before the timed region, for clock samples")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other configurations timed after the default workload")
    ap.add_argument("--config-steps", type=int, default=300,
                    help="back-to-back steps timed for each other configuration")
    return ap.parse_args(argv)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate_max(value: float, world: int, device=None) -> float:
    """Max of `value` over ranks (identity without a process group)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step: int, steps: int, world: int, max_seconds: float) -> float:
    """Units all ranks processed / max-over-ranks time, in GB/s."""
    return bytes_per_step * steps * world / max_seconds / 1e9


def percentile(xs, q):
    xs = sorted(xs)
    if not xs:
        return float("nan")
    k = (len(xs) - 1) * q
    lo, hi = math.floor(k), math.ceil(k)
    return xs[lo] + (xs[hi] - xs[lo]) * (k - lo)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# The sources the fused decode kernel and its host launch are built from.
FUSED_SOURCES = ("cfa_api.cu", "cfa_device.cuh", "cfa_internal.h", "cfa_kernel.cuh", "cfa_merge.cuh",
                 "cfa_kernels_d128.cu", "cfa_kernels_d64.cu", "cfa_tile.cuh")


def kernel_source_digest() -> str:
    """Digest of the fused kernel's CUDA sources; ncu traffic figures are tied to it."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "out_proj_block_gb300", "csrc")
    for name in FUSED_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, cluster_size: int):
    """DRAM bytes per launch from a committed ncu summary of the same kernel
    sources, workload and cluster size, or None."""
    pat = re.compile(r"^traffic_bytes_per_launch:\s*(\d+)\s+workload=(\S+)\s+cluster_size=(\d+)"
                     r"\s+source_digest=(\w+)", re.M)
    digest = kernel_source_digest()
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for name in sorted(os.listdir(pdir)):
        if not name.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, name)) as f:
            for m in pat.finditer(f.read()):
                if m.group(2) == workload and int(m.group(3)) == cluster_size and m.group(4) == digest:
                    return int(m.group(1))
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)
        return summarize_clocks(self.lines)


def summarize_clocks(lines):
    """Median SM clock, max clock and the throttle reasons seen in the samples."""
    sm, smax, reasons, power = [], [], set(), []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            smax.append(float(parts[2]))
            power.append(float(parts[3]))
        except ValueError:
            continue
        for name, val in zip(REASON_NAMES, parts[5:9]):
            if val.lower() == "active":
                reasons.add(name)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
            "reasons": sorted(reasons), "samples": len(sm),
            "power_w_max": max(power) if power else None}


def oracle_baseline(wl, cpu_inputs, budget_s: float, max_reps: int = 50):
    """The fp64 oracle, as it is, on all host cores: full decode steps of the
    workload, repeated until the time budget is spent (at least one)."""
    from oracle import cfa_oracle
    cores = os.cpu_count() or 1
    used = cfa_oracle.threads_used(cores)
    times, ref = [], None
    t_start = time.perf_counter()
    while len(times) < max_reps:
        t0 = time.perf_counter()
        ref = cfa_oracle.decode_step_ex(cpu_inputs["x"], cpu_inputs["W_qkv"], cpu_inputs["W_o"],
                                        cpu_inputs["k_cache"], cpu_inputs["v_cache"],
                                        list(wl.lens), rope_theta=wl.rope_theta, nthreads=used)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start >= budget_s:
            break
    step_s = statistics.median(times)
    # The same oracle on one thread: three full steps, the median.
    one = []
    for _ in range(3):
        t0 = time.perf_counter()
        cfa_oracle.decode_step_ex(cpu_inputs["x"], cpu_inputs["W_qkv"], cpu_inputs["W_o"],
                                  cpu_inputs["k_cache"], cpu_inputs["v_cache"], list(wl.lens),
                                  rope_theta=wl.rope_theta, nthreads=1)
        one.append(time.perf_counter() - t0)
    one_s = statistics.median(one)
    return {"value": wl.algorithmic_bytes / step_s / 1e9, "unit": "GB/s", "cores": used,
            "kind": "oracle",
            "sample": f"{len(times)} full fp64 decode steps of {wl.name} "
                      f"(median {step_s * 1e3:.1f} ms per step)",
            "step_ms": step_s * 1e3,
            "single_thread": {"value": wl.algorithmic_bytes / one_s / 1e9, "unit": "GB/s",
                              "cores": 1, "step_ms": one_s * 1e3,
                              "sample": "3 full fp64 decode steps on one thread, median"}}, ref


# --------------------------------------------------------- reference arm


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import torch
    from out_proj_block_gb300 import workloads
    from oracle import cfa_oracle
    cfa_oracle.build()
    wl = workloads.WORKLOADS[args.workload]
    t = workloads.make_inputs(wl, seed=0, device="cpu")
    cores = os.cpu_count() or 1
    used = cfa_oracle.threads_used(cores)
    run = lambda: cfa_oracle.decode_step_ex(t["x"], t["W_qkv"], t["W_o"], t["k_cache"],
                                            t["v_cache"], list(wl.lens), rope_theta=wl.rope_theta,
                                            nthreads=used)
    for _ in range(max(args.warmup, 0)):
        run()
    times = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        s = time.perf_counter()
        run()
        times.append(time.perf_counter() - s)
    total = time.perf_counter() - t0
    value = wl.algorithmic_bytes * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(wl.as_config(), l2="host run; no GPU L2 involved"),
        "latency_us": {"p50": percentile(times, 0.5) * 1e6, "p10": percentile(times, 0.1) * 1e6,
                       "p90": percentile(times, 0.9) * 1e6},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": used, "kind": "oracle",
                         "sample": f"{args.steps} full fp64 decode steps of {wl.name}"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    del torch
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm


SECONDARY_WORKLOADS = ("llama7b_b1_ctx1k", "llama7b_b16_ctx4k", "llama7b_b1_ctx16k_spiky",
                       "hd64_b8_ctx2k")
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e, nominal


def _fused_plan_and_step(cfa, workloads, wl, dev, n_copies, cluster_size=None, stages=None):
    """Inputs (n_copies rotating sets), a plan and a step(i, stream) callable."""
    import torch
    B, H = wl.B, wl.hidden
    copies = [workloads.make_inputs(wl, seed=i, device=dev) for i in range(max(n_copies, 1))]
    outs = [torch.empty(B, H, dtype=torch.bfloat16, device=dev) for _ in copies]
    plan = cfa.Plan(B, H, wl.n_heads, wl.head_dim, wl.max_ctx,
                    cluster_size=cluster_size, stages=stages)
    uniform = wl.ctx_lens is None and wl.rope_theta == 0.0

    def step(i, stream):
        c = copies[i % len(copies)]
        if uniform:
            plan.decode_step(c["x"], c["W_qkv"], c["W_o"], c["k_cache"], c["v_cache"],
                             wl.ctx_len, outs[i % len(copies)], stream)
        else:
            plan.decode_step_ex(c["x"], c["W_qkv"], c["W_o"], c["k_cache"], c["v_cache"],
                                list(wl.lens), outs[i % len(copies)], wl.rope_theta, stream)

    return copies, outs, plan, step, uniform


def _per_step_ms(step, n, stream, dev):
    """n steps with an event recorded after each; per-step device times in ms."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    ev[0].record(stream)
    for k in range(n):
        step(k, stream)
        ev[k + 1].record(stream)
    torch.cuda.synchronize(dev)
    return [ev[k].elapsed_time(ev[k + 1]) for k in range(n)]


def _back_to_back_s(step, K, stream, dev):
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for k in range(K):
        step(k, stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / 1e3


def _serial_ms(plan, step, n, stream, dev):
    """The kernel-alone step time in ms: n steps with launch overlap off (each
    starts only after the previous step's kernels have finished) between one
    pair of events, so nothing overlaps and no event sits between steps. This
    is the launch's own duration plus the gap between launches, the quantity
    ncu reports as gpu__time_duration per launch. Overlap is restored afterwards."""
    plan.set_overlap(False)
    try:
        for k in range(3):
            step(k, stream)
        ms = _back_to_back_s(step, n, stream, dev) * 1e3 / n
    finally:
        plan.set_overlap(True)
    return ms


def _kernel_only_ms(plan, step, n, stream, dev):
    """Per-step device times with launch overlap off: each step starts only
    after the previous kernel has finished, so an event pair brackets exactly
    one step's kernels (the fused kernel, plus the head merge where the plan
    uses one). n samples; overlap is restored afterwards. Event timestamps on
    this GPU advance in steps of about 1 us, so the mean of many pairs (not a
    percentile) is the estimate; an event between steps adds about 2 us to
    each (compare _serial_ms)."""
    plan.set_overlap(False)
    try:
        for k in range(3):
            step(k, stream)
        ms = _per_step_ms(step, n, stream, dev)
    finally:
        plan.set_overlap(True)
    return ms


def _parity_vs_oracle(wl, copy0, out0, step, stream, dev, nthreads):
    """Copy 0's step recomputed on the GPU and compared with the fp64 oracle
    (out and the appended K/V rows)."""
    import numpy as np
    import torch
    from oracle import cfa_oracle
    cfa_oracle.build()
    cpu = {k: v.cpu() for k, v in copy0.items()}
    ref = cfa_oracle.decode_step_ex(cpu["x"], cpu["W_qkv"], cpu["W_o"], cpu["k_cache"],
                                    cpu["v_cache"], list(wl.lens), rope_theta=wl.rope_theta,
                                    nthreads=nthreads)
    step(0, stream)
    torch.cuda.synchronize(dev)
    got = out0.double().cpu().numpy()
    res = {"out_rel_l2": float(np.linalg.norm(got - ref["out"]) / np.linalg.norm(ref["out"])),
           "out_max_abs": float(np.abs(got - ref["out"]).max())}
    bidx = torch.arange(wl.B)
    rows = torch.tensor(list(wl.lens))
    for name, key in (("k_new", "k_cache"), ("v_new", "v_cache")):
        g = copy0[key].cpu()[bidx, :, rows].double().numpy()
        r = ref[name]
        res[f"{name}_rel_l2"] = float(np.linalg.norm(g - r) / np.linalg.norm(r))
        res[f"{name}_max_abs"] = float(np.abs(g - r).max())
    return res


def measure_secondary(cfa, workloads, name, dev, steps, peak, nthreads, with_parity):
    """One more workload on the same GPU: back-to-back and kernel-only
    per-step time, GB/s, roofline fractions and parity against the oracle."""
    import torch
    wl = workloads.WORKLOADS[name]
    n_copies = max(2, -(-300_000_000 // wl.algorithmic_bytes))  # rotate > 2x the L2
    copies, outs, plan, step, _ = _fused_plan_and_step(cfa, workloads, wl, dev, n_copies)
    stream = torch.cuda.current_stream(dev)
    try:
        desc = plan.describe()
        for k in range(10):
            step(k, stream)
        torch.cuda.synchronize(dev)
        total_s = _back_to_back_s(step, steps, stream, dev)
        k_us = _serial_ms(plan, step, 300, stream, dev) * 1e3
        kern = _kernel_only_ms(plan, step, 300, stream, dev)
        if plan.status() != cfa.CFA_OK:
            raise RuntimeError(f"{name}: device status after timing")
        b2b_us = total_s / steps * 1e6
        res = {"workload": name, "B": wl.B, "ctx_len": wl.ctx_len, "head_dim": wl.head_dim,
               "n_heads": wl.n_heads, "cluster_size": desc["cluster_size"],
               "stages": desc["stages"], "launches_per_step": desc["launches_per_step"],
               "algorithmic_bytes": wl.algorithmic_bytes,
               "us_per_step_back_to_back": b2b_us, "us_per_step_kernel": k_us,
               "us_per_step_kernel_event_pairs": statistics.fmean(kern) * 1e3,
               "gbs_back_to_back": wl.algorithmic_bytes / b2b_us / 1e3,
               "gbs_kernel": wl.algorithmic_bytes / k_us / 1e3,
               "frac_kernel": wl.algorithmic_bytes / k_us / 1e3 / peak,
               "frac_pipelined": wl.algorithmic_bytes / b2b_us / 1e3 / peak,
               "steps": steps, "kernel_samples": len(kern), "input_copies": n_copies}
        if with_parity:
            res["parity"] = _parity_vs_oracle(wl, copies[0], outs[0], step, stream, dev, nthreads)
        return res
    finally:
        plan.close()
        del copies, outs
        torch.cuda.empty_cache()


def run_ours(args):
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    from out_proj_block_gb300 import build as cuda_build
    if rank == 0 or world == 1:
        cuda_build.build()
    if world > 1:
        torch.distributed.barrier()
    from out_proj_block_gb300 import cfa, workloads

    wl = workloads.WORKLOADS[args.workload]
    B, H = wl.B, wl.hidden
    copies, outs, plan, step, uniform = _fused_plan_and_step(
        cfa, workloads, wl, dev, args.copies, args.cluster_size, args.stages)
    desc = plan.describe()
    stream = torch.cuda.current_stream(dev)

    for i in range(max(args.warmup, 3)):
        step(i, stream)
    torch.cuda.synchronize(dev)
    st = plan.status()
    if st != cfa.CFA_OK:
        raise RuntimeError(f"device status after warm-up: {cfa.cfa_status_string(st)}")

    sampler = ClockSampler(local).start()
    t_end = time.perf_counter() + args.preload_seconds
    i = 0
    while time.perf_counter() < t_end:  # untimed load so clocks settle and get sampled
        for _ in range(64):
            step(i, stream)
            i += 1
        torch.cuda.synchronize(dev)

    K = args.steps
    if world > 1:
        torch.distributed.barrier()
    total_s = _back_to_back_s(step, K, stream, dev)
    if world > 1:
        torch.distributed.barrier()
    # Kernel-alone time (launch overlap off): serialised steps between one
    # pair of events, and per-step event pairs beside it; at least 300 / 400
    # steps whatever K is.
    n_serial = max(300, min(K, 2000))
    serial_ms = _serial_ms(plan, step, n_serial, stream, dev)
    n_kern = max(400, min(K, 2000))
    kern_ms = _kernel_only_ms(plan, step, n_kern, stream, dev)
    clocks = sampler.stop()
    st = plan.status()
    if st != cfa.CFA_OK:
        raise RuntimeError(f"device status after timing: {cfa.cfa_status_string(st)}")

    # Per-step latency with overlap on and an event between steps (untimed for
    # the headline).
    n_iso = max(200, min(K, 500))
    step_ms = _per_step_ms(step, n_iso, stream, dev)
    max_total_s = aggregate_max(total_s, world, dev)
    value = whole_job_gbs(wl.algorithmic_bytes, K, world, max_total_s)
    mean_step_s = total_s / K
    kernel_s = serial_ms / 1e3

    # CUDA-graph replay of the same steps (launch overhead removed)
    graph_us = None
    try:
        g = torch.cuda.CUDAGraph()
        s2 = torch.cuda.Stream(dev)
        s2.wait_stream(stream)
        with torch.cuda.stream(s2):
            with torch.cuda.graph(g, stream=s2):
                for k in range(len(copies)):
                    step(k, s2)
        stream.wait_stream(s2)
        reps = max(1, max(K, 300) // len(copies))
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        graph_us = e0.elapsed_time(e1) * 1e3 / (reps * len(copies))
    except Exception as exc:  # graph capture is an extra measurement, not the headline
        graph_us = f"unavailable: {type(exc).__name__}: {exc}"

    # end-to-end through the host-buffer entry point
    e2e = None
    if not args.no_e2e and uniform:
        x_host = [c["x"].cpu().pin_memory() for c in copies]
        out_host = [torch.empty(B, H, dtype=torch.bfloat16).pin_memory() for _ in copies]

        def host_step(k):
            c = copies[k % len(copies)]
            plan.decode_step_host(x_host[k % len(copies)], c["W_qkv"], c["W_o"], c["k_cache"],
                                  c["v_cache"], wl.ctx_len, out_host[k % len(copies)], stream)

        for k in range(max(args.warmup, 3)):
            host_step(k)
        if world > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        for k in range(K):
            host_step(k)
        e2e_s = aggregate_max(time.perf_counter() - t0, world, dev)
        e2e = {"value": whole_job_gbs(wl.algorithmic_bytes, K, world, e2e_s), "unit": "GB/s",
               "h2d_bytes_per_step": int(x_host[0].numel() * 2),
               "d2h_bytes_per_step": int(out_host[0].numel() * 2),
               "ms_per_step": e2e_s / K * 1e3}

    peak, peak_kind = measured_peaks()
    achieved = wl.algorithmic_bytes / kernel_s / 1e9
    achieved_pipe = wl.algorithmic_bytes / mean_step_s / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
            "traffic": recorded_traffic(wl.name, plan.cluster_size),
            "algorithmic_bytes_per_launch": wl.algorithmic_bytes,
            "kernel": "cfa::fused_decode_kernel",
            "duration_us": kernel_s * 1e6,
            "duration_source": f"{n_serial} steps with launch overlap off (each starts after "
                               "the previous one's kernels have finished) between one pair of "
                               "CUDA events on the launching stream, divided by the step count: "
                               "the launch's own duration plus the gap between launches, as ncu "
                               "gpu__time_duration measures it; with an event pair around each "
                               f"step instead the mean is {statistics.fmean(kern_ms) * 1e3:.2f} us"
                               + ("; the step is this kernel plus the head-merge kernel"
                                  if desc.get("launches_per_step", 1) > 1 else ""),
            "achieved_pipelined": achieved_pipe, "frac_pipelined": achieved_pipe / peak,
            "pipelined_note": "back-to-back steps whose launches overlap (programmatic "
                              "dependent launch): the next step's prologue and first weight "
                              "loads run under this step's tail",
            "frac_vs_nominal": achieved / NOMINAL_HBM_GBS, "nominal_gbs": NOMINAL_HBM_GBS}

    cpu_base, parity = None, None
    nthreads = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_inputs = {k: v.cpu() for k, v in copies[0].items()}
        cpu_base, ref = oracle_baseline(wl, cpu_inputs, args.cpu_seconds)
        nthreads = cpu_base["cores"]
        parity = _parity_vs_oracle(wl, copies[0], outs[0], step, stream, dev, nthreads)

    plan.close()
    del copies, outs
    torch.cuda.empty_cache()

    # The other configurations of the block, after the headline.
    configs = None
    if rank == 0 and world == 1 and not args.no_configs and args.workload == DEFAULT_WORKLOAD:
        configs = []
        for name in SECONDARY_WORKLOADS:
            configs.append(measure_secondary(cfa, workloads, name, dev, args.config_steps, peak,
                                             nthreads or (os.cpu_count() or 1),
                                             not args.no_cpu_baseline))

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": max_total_s / K * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": dict(wl.as_config(), cluster_size=desc["cluster_size"],
                       stages=desc["stages"], grid=desc["grid"],
                       l2=f"{args.copies} rotating input copies of "
                          f"{wl.algorithmic_bytes / 1e6:.0f} MB each (> 129 MB L2)",
                       parallelism=f"replicas x{world}"),
        "latency_us": {"back_to_back_mean": mean_step_s * 1e6,
                       "kernel": serial_ms * 1e3,
                       "kernel_event_pairs_mean": statistics.fmean(kern_ms) * 1e3,
                       "kernel_p10": percentile(kern_ms, 0.1) * 1e3,
                       "kernel_p50": percentile(kern_ms, 0.5) * 1e3,
                       "kernel_p90": percentile(kern_ms, 0.9) * 1e3,
                       "kernel_samples": len(kern_ms),
                       "isolated_p10": percentile(step_ms, 0.1) * 1e3,
                       "isolated_p50": percentile(step_ms, 0.5) * 1e3,
                       "isolated_p90": percentile(step_ms, 0.9) * 1e3,
                       "isolated_samples": len(step_ms),
                       "note": "back_to_back: K steps between two events (consecutive steps "
                               "overlap via programmatic dependent launch); kernel: steps with "
                               "launch overlap off between one pair of events, per step; "
                               "kernel_event_pairs / kernel_p*: one step between two events "
                               "with launch overlap off; isolated: an event after every step, "
                               "overlap on"},
        "graph_latency_us": graph_us,
        "roofline": roof,
        "cpu_baseline": cpu_base,
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": K * desc.get("launches_per_step", 1),
        "parity": parity,
        "configs": configs,
        "plan": desc,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


# ------------------------------------------------- the decode loop (stack)


def stack_oracle_tokens(wl, t_cpu, budget_s: float, max_tokens: int = 20):
    """The fp64 oracle stack on all host cores, one token (every layer) at a
    time until the budget is spent (at least one)."""
    import numpy as np
    import torch
    from oracle import cfa_oracle
    cfa_oracle.build()
    cores = os.cpu_count() or 1
    used = cfa_oracle.threads_used(cores)
    caches = [(l["k_cache"].view(torch.int16).numpy().view(np.uint16).copy(),
               l["v_cache"].view(torch.int16).numpy().view(np.uint16).copy())
              for l in t_cpu["layers"]]
    times, y = [], None
    t_start = time.perf_counter()
    while len(times) < max_tokens:
        t0 = time.perf_counter()
        y, _ = cfa_oracle.stack_step(t_cpu["x"], t_cpu["layers"], caches, list(wl.lens),
                                     wl.rope_theta, wl.eps, used)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start >= budget_s:
            break
    return times, used, y


def run_stack_reference(args, wl):
    import torch
    from out_proj_block_gb300 import workloads
    t = workloads.make_stack_inputs(wl, seed=0, device="cpu")
    budget = 1e9  # the reference arm runs exactly warmup + steps tokens
    for _ in range(max(args.warmup, 0)):
        stack_oracle_tokens(wl, t, 0.0, max_tokens=1)
    t0 = time.perf_counter()
    times, used, _ = stack_oracle_tokens(wl, t, budget, max_tokens=args.steps)
    total = time.perf_counter() - t0
    value = wl.algorithmic_bytes * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(wl.as_config(), l2="host run; no GPU L2 involved"),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": used, "kind": "oracle",
                         "sample": f"{args.steps} tokens through all {wl.n_layers} layers"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    del torch
    print(json.dumps(line), flush=True)
    return 0


def run_stack(args, wl):
    """The decode loop: one token through every layer per step, from a graph."""
    import numpy as np
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from out_proj_block_gb300 import build as cuda_build
    if rank == 0 or world == 1:
        cuda_build.build()
    if world > 1:
        torch.distributed.barrier()
    from out_proj_block_gb300 import cfa, workloads

    t = workloads.make_stack_inputs(wl, seed=0, device=dev)
    stack = cfa.Stack(wl.n_layers, wl.B, wl.hidden, wl.n_heads, wl.head_dim, wl.ffn, wl.max_ctx,
                      layers=t["layers"])
    desc = stack.describe()
    pos = torch.tensor(list(wl.lens), dtype=torch.int32, device=dev)
    x = t["x"]
    out = torch.empty_like(x)
    stream = torch.cuda.Stream(dev)
    launches_per_token = desc["launches_per_token"]

    def token(graph=True):
        (stack.step_graph if graph else stack.step)(x, pos, out, wl.rope_theta, wl.eps,
                                                    advance=False, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            token()
    torch.cuda.synchronize(dev)
    st = stack.status()
    if st != cfa.CFA_OK:
        raise RuntimeError(f"device status after warm-up: {cfa.cfa_status_string(st)}")

    sampler = ClockSampler(local).start()
    t_end = time.perf_counter() + args.preload_seconds
    with torch.cuda.stream(stream):
        while time.perf_counter() < t_end:
            for _ in range(8):
                token()
            torch.cuda.synchronize(dev)
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(K):
            token()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    total_s = e0.elapsed_time(e1) / 1e3
    st = stack.status()
    if st != cfa.CFA_OK:
        raise RuntimeError(f"device status after timing: {cfa.cfa_status_string(st)}")
    max_total_s = aggregate_max(total_s, world, dev)
    value = whole_job_gbs(wl.algorithmic_bytes, K, world, max_total_s)
    mean_s = total_s / K

    # per-token latency with an event after every token, and eager launches
    n_iso = min(K, 100)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_iso + 1)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for k in range(n_iso):
            token()
            ev[k + 1].record(stream)
    torch.cuda.synchronize(dev)
    tok_ms = [ev[k].elapsed_time(ev[k + 1]) for k in range(n_iso)]
    n_eager = min(K, 100)
    with torch.cuda.stream(stream):
        token(graph=False)
        e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2.record(stream)
        for _ in range(n_eager):
            token(graph=False)
        e3.record(stream)
    torch.cuda.synchronize(dev)
    eager_ms = e2.elapsed_time(e3) / n_eager

    # end to end: pinned host x in, pinned host out back, every token
    e2e = None
    if not args.no_e2e:
        x_host = x.cpu().pin_memory()
        out_host = torch.empty(x.shape, dtype=torch.bfloat16).pin_memory()
        x_dev = torch.empty_like(x)

        def host_token():
            with torch.cuda.stream(stream):
                x_dev.copy_(x_host, non_blocking=True)
                stack.step_graph(x_dev, pos, out, wl.rope_theta, wl.eps, advance=False,
                                 stream=stream)
                out_host.copy_(out, non_blocking=True)
            stream.synchronize()

        for _ in range(3):
            host_token()
        n_e2e = min(K, 200)
        if world > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            host_token()
        e2e_s = aggregate_max(time.perf_counter() - t0, world, dev)
        e2e = {"value": whole_job_gbs(wl.algorithmic_bytes, n_e2e, world, e2e_s), "unit": "GB/s",
               "h2d_bytes_per_step": int(x_host.numel() * 2),
               "d2h_bytes_per_step": int(out_host.numel() * 2),
               "ms_per_step": e2e_s / n_e2e * 1e3, "steps": n_e2e}

    peak, peak_kind = measured_peaks()
    achieved = wl.algorithmic_bytes / mean_s / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs", "traffic": None,
            "algorithmic_bytes_per_launch": wl.algorithmic_bytes,
            "kernel": f"whole token ({launches_per_token} kernels from one graph launch)"}

    cpu_base, parity = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t_cpu = {"x": x.cpu(), "layers": [{k: v.cpu() for k, v in l.items()} for l in t["layers"]]}
        times, used, y_ref = stack_oracle_tokens(wl, t_cpu, args.cpu_seconds)
        tok_s = statistics.median(times)
        cpu_base = {"value": wl.algorithmic_bytes / tok_s / 1e9, "unit": "GB/s", "cores": used,
                    "kind": "oracle",
                    "sample": f"{len(times)} fp64 tokens through all {wl.n_layers} layers "
                              f"(median {tok_s * 1e3:.0f} ms per token)",
                    "step_ms": tok_s * 1e3}
        got = out.double().cpu().numpy()
        ref = (np.ascontiguousarray(y_ref).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        parity = {"out_rel_l2": float(np.linalg.norm(got - ref) / np.linalg.norm(ref)),
                  "out_max_abs": float(np.abs(got - ref).max())}

    stack.close()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": max_total_s / K * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": dict(wl.as_config(),
                       l2=f"one token reads {wl.algorithmic_bytes / 1e9:.1f} GB (> 129 MB L2)",
                       parallelism=f"replicas x{world}"),
        "latency_us": {"graph_back_to_back_mean": mean_s * 1e6,
                       "graph_isolated_p10": percentile(tok_ms, 0.1) * 1e3,
                       "graph_isolated_p50": percentile(tok_ms, 0.5) * 1e3,
                       "graph_isolated_p90": percentile(tok_ms, 0.9) * 1e3,
                       "eager_mean": eager_ms * 1e3},
        "roofline": roof,
        "cpu_baseline": cpu_base,
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": K * launches_per_token,
        "parity": parity,
        "plan": desc,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


# ------------------------------------------- multi-head latent attention


def mla_oracle_steps(wl, t_cpu, budget_s: float, max_steps: int = 20):
    """The fp64 MLA oracle on all host cores, whole steps until the budget is spent."""
    from oracle import cfa_oracle
    cfa_oracle.build()
    used = cfa_oracle.threads_used(os.cpu_count() or 1)
    times, ref = [], None
    t_start = time.perf_counter()
    while len(times) < max_steps:
        t0 = time.perf_counter()
        ref = cfa_oracle.mla_step(t_cpu["x"], t_cpu["W_a"], t_cpu["g_q"], t_cpu["g_kv"],
                                  t_cpu["W_uq"], t_cpu["W_kvb"], t_cpu["W_o"], t_cpu["cache"],
                                  list(wl.lens), wl.rope_theta, wl.eps, used)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start >= budget_s:
            break
    return times, used, ref


def run_mla_reference(args, wl):
    from out_proj_block_gb300 import workloads
    t = workloads.make_mla_inputs(wl, seed=0, device="cpu")
    for _ in range(max(args.warmup, 0)):
        mla_oracle_steps(wl, t, 0.0, max_steps=1)
    t0 = time.perf_counter()
    times, used, _ = mla_oracle_steps(wl, t, 1e9, max_steps=args.steps)
    total = time.perf_counter() - t0
    value = wl.algorithmic_bytes * args.steps / total / 1e9
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(wl.as_config(), l2="host run; no GPU L2 involved"),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": used, "kind": "oracle",
                         "sample": f"{args.steps} full fp64 MLA steps of {wl.name}"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0}), flush=True)
    return 0


def run_mla(args, wl):
    """MLA decode steps (4 launches each) back to back."""
    import numpy as np
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from out_proj_block_gb300 import build as cuda_build
    if rank == 0 or world == 1:
        cuda_build.build()
    if world > 1:
        torch.distributed.barrier()
    from out_proj_block_gb300 import cfa, workloads

    t = workloads.make_mla_inputs(wl, seed=0, device=dev)
    mla = cfa.Mla(wl.B, wl.hidden, wl.n_heads, wl.q_lora, wl.max_ctx)
    desc = mla.describe()
    out = torch.empty(wl.B, wl.hidden, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    lens = list(wl.lens)

    def step():
        mla.step(t["x"], t, t["cache"], lens, out, wl.rope_theta, wl.eps, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    if mla.status() != cfa.CFA_OK:
        raise RuntimeError("device status after warm-up")
    sampler = ClockSampler(local).start()
    t_end = time.perf_counter() + args.preload_seconds
    while time.perf_counter() < t_end:
        for _ in range(32):
            step()
        torch.cuda.synchronize(dev)
    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    total_s = e0.elapsed_time(e1) / 1e3
    if mla.status() != cfa.CFA_OK:
        raise RuntimeError("device status after timing")
    max_total_s = aggregate_max(total_s, world, dev)
    value = whole_job_gbs(wl.algorithmic_bytes, K, world, max_total_s)
    mean_s = total_s / K
    n_iso = min(K, 200)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_iso + 1)]
    ev[0].record(stream)
    for k in range(n_iso):
        step()
        ev[k + 1].record(stream)
    torch.cuda.synchronize(dev)
    step_ms = [ev[k].elapsed_time(ev[k + 1]) for k in range(n_iso)]

    e2e = None
    if not args.no_e2e:
        x_host = t["x"].cpu().pin_memory()
        out_host = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
        x_dev = torch.empty_like(t["x"])

        def host_step():
            x_dev.copy_(x_host, non_blocking=True)
            mla.step(x_dev, t, t["cache"], lens, out, wl.rope_theta, wl.eps, stream)
            out_host.copy_(out, non_blocking=True)
            stream.synchronize()

        for _ in range(3):
            host_step()
        n_e2e = min(K, 500)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            host_step()
        e2e_s = aggregate_max(time.perf_counter() - t0, world, dev)
        e2e = {"value": whole_job_gbs(wl.algorithmic_bytes, n_e2e, world, e2e_s), "unit": "GB/s",
               "h2d_bytes_per_step": int(x_host.numel() * 2),
               "d2h_bytes_per_step": int(out_host.numel() * 2),
               "ms_per_step": e2e_s / n_e2e * 1e3, "steps": n_e2e}

    peak, peak_kind = measured_peaks()
    achieved = wl.algorithmic_bytes / mean_s / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs", "traffic": None,
            "algorithmic_bytes_per_launch": wl.algorithmic_bytes,
            "kernel": "whole MLA step (4 kernels)",
            "attention_flops_per_step": wl.attention_flops}
    cpu_base, parity = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t_cpu = {k: v.cpu() for k, v in t.items()}
        times, used, ref = mla_oracle_steps(wl, t_cpu, args.cpu_seconds)
        st_s = statistics.median(times)
        cpu_base = {"value": wl.algorithmic_bytes / st_s / 1e9, "unit": "GB/s", "cores": used,
                    "kind": "oracle",
                    "sample": f"{len(times)} full fp64 MLA steps of {wl.name} "
                              f"(median {st_s * 1e3:.0f} ms per step)", "step_ms": st_s * 1e3}
        step()
        torch.cuda.synchronize(dev)
        got = out.double().cpu().numpy()
        parity = {"out_rel_l2": float(np.linalg.norm(got - ref["out"]) / np.linalg.norm(ref["out"])),
                  "out_max_abs": float(np.abs(got - ref["out"]).max())}
    mla.close()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": max_total_s / K * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": dict(wl.as_config(),
                       l2=f"one step reads {wl.algorithmic_bytes / 1e6:.0f} MB (> 129 MB L2)",
                       parallelism=f"replicas x{world}"),
        "latency_us": {"back_to_back_mean": mean_s * 1e6,
                       "isolated_p10": percentile(step_ms, 0.1) * 1e3,
                       "isolated_p50": percentile(step_ms, 0.5) * 1e3,
                       "isolated_p90": percentile(step_ms, 0.9) * 1e3},
        "roofline": roof, "cpu_baseline": cpu_base, "e2e": e2e, "clocks": clocks,
        "gpu_launches": 4 * K, "parity": parity, "plan": desc,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    from out_proj_block_gb300 import workloads
    if args.workload in workloads.MLAS:
        wl = workloads.MLAS[args.workload]
        if args.impl == "reference":
            world, rank, _ = dist_env()
            return run_mla_reference(args, wl) if rank == 0 else 0
        return run_mla(args, wl)
    if args.workload in workloads.STACKS:
        wl = workloads.STACKS[args.workload]
        if args.impl == "reference":
            world, rank, _ = dist_env()
            return run_stack_reference(args, wl) if rank == 0 else 0
        return run_stack(args, wl)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
