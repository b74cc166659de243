#!/usr/bin/env python
"""Benchmark of the ANVIL optimizer step on GB300: one full step over the three
projection banks (qk 22x256x768, vo 22x768x768, mlp 22x2816x768; 66 matrices), mixed
synthetic inputs (half Gaussian, half rank-32 plus 1e-3 noise), post-engage scalars,
each step one CUDA-graph replay of its four launches (momentum, d, X / d, the cascade).

Prints one JSON line (rank 0).  ``value`` is whole-job matrices/s with the inputs
resident in HBM; ``e2e`` is the same metric through the same C-ABI call with the
gradients copied in from pinned host memory and the outputs copied back every step;
``roofline`` is the dominant kernel's achieved rate (algorithmic work / its CUDA-event
duration inside timed steps) against the measured peak; ``cpu_baseline`` is the CPU
oracle on a bounded sample of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl anvil|reference]
  python bench.py --ncu-case     # two eager steps of the same workload, for ncu captures
  python bench.py --tail-ncu-case  # one step writing the tail link, then the tail without and with it

``--impl reference`` times the CPU oracle (the reference arm: no installable reference exists) on the same
workload and metric.  With N > 1 (launched by torch.distributed.run) every rank runs an
independent replica of the step on its own GPU: the path shards by whole matrices and
has no exchange step, so there is no collective on the data path.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from polynomial_matrix_whitening_gb300 import workloads as W  # noqa: E402

METRIC = "ANVIL bank-step matrices/s and TFLOP/s; % of GB300 bf16 tensor peak"
UNIT = "matrices/s"
WORKLOAD = "full_step"
GEMM_KINDS = ("gram", "gram_norm", "sqpoly", "xupdate", "xupdate_out", "cascade")

# ncu DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of each
# kernel kind on this workload, taken from one ncu capture of the cascade launch of the
# full three-bank step (not measured by this run); valid only while the kernel source
# hashes to the recorded value, reported as null otherwise.
NCU_TRAFFIC = {
    "cascade": {"bytes_per_launch": 2868.7e6, "source_hash": "7c85ec962766be48"},
}


def kernel_source_hash(kind):
    name = "anvil_elementwise.cu" if kind in ("momentum", "norm_d", "normalize") else "anvil_gemm.cu"
    with open(os.path.join(ROOT, "polynomial_matrix_whitening_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ------------------------------------------------------------------ work accounting

def bank_dims(banks):
    out = []
    for b in banks:
        s, L = min(b.m, b.n), max(b.m, b.n)
        out.append((b.g, b.m, b.n, s, L))
    return out


def algorithmic_work(banks, nmaps=6):
    """Per launch of each kernel kind over all banks: flops (GEMMs, symmetric products
    counted on one triangle) or bytes (elementwise kernels)."""
    w = {"gram": 0.0, "gram_norm": 0.0, "sqpoly": 0.0, "xupdate": 0.0, "xupdate_out": 0.0,
         "momentum": 0.0, "normalize": 0.0, "norm_d": 0.0, "cascade": 0.0}
    for g, m, n, s, L in bank_dims(banks):
        w["gram"] += g * s * (s + 1) * L
        w["gram_norm"] += g * s * (s + 1) * L
        w["sqpoly"] += g * s * (s + 1) * s
        w["xupdate"] += g * 2.0 * s * s * L
        w["xupdate_out"] += g * 2.0 * s * s * L
        w["momentum"] += g * m * n * 22.0        # 4 B grad + 2x(4+4) B rails + 2 B X
        w["normalize"] += g * m * n * 4.0        # read + write bf16
        w["norm_d"] += g * m * 4.0
        # the cascade kernel: every product of every map
        w["cascade"] += g * nmaps * (s * (s + 1) * L + s * (s + 1) * s + 2.0 * s * s * L)
    return w


def step_flops(banks, nmaps=6):
    alg = dense = 0.0
    for g, m, n, s, L in bank_dims(banks):
        alg += g * nmaps * (s * (s + 1) * L + s * (s + 1) * s + 2.0 * s * s * L)
        dense += g * nmaps * (4.0 * s * s * L + 2.0 * s ** 3)
    return alg, dense


# ------------------------------------------------------------------ clocks

def physical_gpu(local):
    """The nvidia-smi id (index, UUID or bus id, as CUDA_VISIBLE_DEVICES lists it) of this
    rank's GPU."""
    ids = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    return ids[local] if local < len(ids) else str(local)


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons every 200 ms while running."""
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() in ("active", "1", "0x1"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ distributed plumbing

def dist_setup():
    """Replicas: one process per GPU (NCCL), or gloo when no GPU is present (host tests).
    The collectives are only the barrier and the max-over-ranks of the step time."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return world, rank, local


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(ms_local, mats_per_rank, world):
    """Whole-job matrices/s of independent replicas: every rank's matrices over the
    slowest rank's step time."""
    ms = max_over_ranks(ms_local, world)
    return ms, mats_per_rank * world / (ms / 1000.0)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ the CPU oracle arm

def oracle_sample(wl, per_bank, min_seconds=0.0):
    """Times the oracle on `per_bank` matrices of each bank of the workload (step 0 of the
    grad pool, zero rails; the first of each bank Gaussian, the second rank-32 + noise),
    repeated until at least `min_seconds` of CPU work, and extrapolates the mean time per
    matrix of each bank to matrices/s of the full step."""
    import oracle
    oracle.build()
    picks, samples = [], []
    for j, b in enumerate(wl.banks):
        grad = wl.grad(j, 0)
        idx = [0, b.g // 2][:per_bank] if per_bank <= 2 else list(range(per_bank))
        picks.append(f"{b.name}{list(idx)}")
        samples += [(j, np.ascontiguousarray(grad[i:i + 1])) for i in idx]
    sc = wl.scalars(0)
    times = [[] for _ in wl.banks]
    secs, rounds = 0.0, 0
    while rounds == 0 or secs < min_seconds:
        for j, g1 in samples:
            v1 = np.zeros((2,) + g1.shape, np.float32)
            t0 = time.perf_counter()
            oracle.bank_step(g1, v1, sc.momentum, sc.fast_beta, sc.fast_weight, sc.slow_beta)
            dt = time.perf_counter() - t0
            times[j].append(dt)
            secs += dt
        rounds += 1
    est = sum(b.g * statistics.mean(times[j]) for j, b in enumerate(wl.banks))
    total = sum(b.g for b in wl.banks)
    return total / est, secs, oracle.num_threads(), ", ".join(picks) + f" x {rounds} rounds"


REFERENCE_BUDGET_S = 150.0   # default CPU seconds the reference arm may spend on its warm-up and timed steps


def workload_config(world):
    """The `config` of the bench line, shared by both arms."""
    return {"workload": WORKLOAD,
            "banks": "qk 22x256x768 + vo 22x768x768 + mlp 22x2816x768",
            "inputs": "matrices 0-10 N(0,0.02^2), 11-21 rank-32 + 1e-3 noise; pool of 4",
            "scalars": "post-engage: momentum 0.95, fast_beta 0.85, fast_weight 0.4385, "
                       "slow_beta 0.98",
            "maps": "6 ANVIL_MAPS",
            "graph": "the timed steps captured as one CUDA graph (4 kernels per step)",
            "l2": "inputs larger than L2 (grads 260 MB + rails 520 MB per step)",
            "parallelism": f"replicas x{world}"}


def run_reference(args, world, rank):
    """The CPU oracle on the bench's step: the same banks, grad pool (step s reads pool
    entry s mod 4) and running rails as the GPU arm.  Every step is the whole 66-matrix
    step when the warm-up and timed steps fit REFERENCE_BUDGET_S; otherwise each step takes
    the same number of matrices from every bank (the step's own bank mix), as many as fit.
    (The budget is --reference-budget, default REFERENCE_BUDGET_S.)"""
    if rank != 0:
        return
    import oracle
    oracle.build()
    wl = W.workloads()[WORKLOAD]
    sc = wl.scalars(0)
    scal = (sc.momentum, sc.fast_beta, sc.fast_weight, sc.slow_beta)
    pool = [[wl.grad(j, p) for j in range(len(wl.banks))] for p in range(wl.pool)]
    # cost of one matrix of each bank, to size the step
    t_full = 0.0
    for j, b in enumerate(wl.banks):
        g1 = np.ascontiguousarray(pool[0][j][:1])
        t0 = time.perf_counter()
        oracle.bank_step(g1, np.zeros((2,) + g1.shape, np.float32), *scal)
        t_full += b.g * (time.perf_counter() - t0)
    g_full = min(b.g for b in wl.banks)
    nsteps = args.steps + args.warmup
    budget = args.reference_budget
    per_bank = g_full if nsteps * t_full <= budget else max(1, int(g_full * budget / (nsteps * t_full)))
    vel = [np.zeros((2, per_bank, b.m, b.n), np.float32) for b in wl.banks]

    def step(s):
        for j in range(len(wl.banks)):
            grad = np.ascontiguousarray(pool[s % wl.pool][j][:per_bank])
            _, vel[j] = oracle.bank_step(grad, vel[j], *scal)

    for s in range(args.warmup):
        step(s)
    t0 = time.perf_counter()
    for s in range(args.steps):
        step(s)
    wall = time.perf_counter() - t0
    mats = per_bank * len(wl.banks) * args.steps
    value = mats / wall
    ms = 1000.0 * wall / args.steps
    whole = per_bank == g_full
    sample = (f"{'the whole step' if whole else f'{per_bank} matrices of each bank per step'} "
              f"({per_bank * len(wl.banks)} matrices: {per_bank} per bank, pool entry s mod 4, running "
              f"rails), {args.steps} timed steps in {wall:.1f} s after {args.warmup} warm-up steps")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(world),
        "matrices_per_step": per_bank * len(wl.banks),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------------ the GPU arm

def run_anvil(args, world, rank, local):
    import torch
    from polynomial_matrix_whitening_gb300 import anvil

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = W.workloads()[WORKLOAD]
    sc = wl.scalars(0)
    scal = dict(momentum=sc.momentum, fast_beta=sc.fast_beta, fast_weight=sc.fast_weight,
                slow_beta=sc.slow_beta)
    pool_h = [[wl.grad(j, p) for j in range(len(wl.banks))] for p in range(wl.pool)]
    pool_d = [[torch.from_numpy(x).to(dev) for x in p] for p in pool_h]
    banks = [anvil.Bank(pool_d[0][j], torch.from_numpy(wl.velocity(j)).to(dev),
                        torch.empty((b.g, b.m, b.n), dtype=torch.bfloat16, device=dev), **scal)
             for j, b in enumerate(wl.banks)]
    shapes = [b.shape for b in banks]
    ws = anvil.alloc_workspace(shapes, device=dev)
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())

    def capture(grads):
        for b, gt in zip(banks, grads):
            b.grad = gt
        anvil.multi_bank_step(banks, ws, stream=stream)  # outside capture: device set-up
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            anvil.multi_bank_step(banks, ws, stream=stream)
        return gr

    launches_per_step = 4   # momentum, norm_d, normalize, the cascade
    nsteps, nwarm = args.steps, args.warmup

    def capture_sequence(count):
        """One CUDA graph of `count` consecutive steps, step s reading pool entry s mod 4."""
        for b, gt in zip(banks, pool_d[0]):
            b.grad = gt
        anvil.multi_bank_step(banks, ws, stream=stream)  # outside capture: device set-up
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for s in range(count):
                for b, gt in zip(banks, pool_d[s % wl.pool]):
                    b.grad = gt
                anvil.multi_bank_step(banks, ws, stream=stream)
        return gr

    # ---- timed region: the K steps as one graph (chunks of at most 1000 steps),
    # inputs resident in HBM
    chunk = min(nsteps, 1000)
    with torch.cuda.stream(stream):
        seq = capture_sequence(chunk)
        warm = capture_sequence(nwarm)
        rest = capture_sequence(nsteps % chunk) if nsteps % chunk else None
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        warm.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    sampler = ClockSampler(physical_gpu(local))
    with sampler, torch.cuda.stream(stream):
        time.sleep(0.25)
        e0.record(stream)
        for _ in range(nsteps // chunk):
            seq.replay()
        if rest is not None:
            rest.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    del seq, warm, rest
    ms = e0.elapsed_time(e1) / nsteps
    clocks = sampler.summary()
    # Peak for the tensor-bound kernel: the burst cuBLAS figure unless the GPU hit its power
    # cap during the timed region (then the sustained figure); with no clock samples, a
    # timed region of a second or more counts as sustained.
    power_capped = ("sw_power_cap" in clocks["reasons"]) if clocks else ms * nsteps >= 1000.0
    mats = sum(b.shape[0] for b in banks)
    ms_max, value = job_value(ms, mats, world)
    alg, dense = step_flops(wl.banks)

    # ---- per-kernel CUDA-event durations over timed steps (same launches, not in a graph)
    prof_steps = max(3, min(nsteps, 20))
    with torch.cuda.stream(stream):
        for s in range(2):
            for b, gt in zip(banks, pool_d[s % wl.pool]):
                b.grad = gt
            anvil.multi_bank_step(banks, ws, stream=stream)
        torch.cuda.synchronize()
        with anvil.profile(max_records=prof_steps * launches_per_step + 8) as prof:
            p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            p0.record(stream)
            for s in range(prof_steps):
                for b, gt in zip(banks, pool_d[s % wl.pool]):
                    b.grad = gt
                anvil.multi_bank_step(banks, ws, stream=stream)
            p1.record(stream)
    torch.cuda.synchronize()
    prof_ms_step = p0.elapsed_time(p1) / prof_steps
    work = algorithmic_work(wl.banks)
    peaks = measured_peaks()
    per_kind = {}
    for kind, t in prof.records:
        d = per_kind.setdefault(kind, [0, 0.0])
        d[0] += 1
        d[1] += t
    tensor_peak = peaks["bf16_tflops_sustained"] if power_capped else peaks["bf16_tflops"]
    tensor_peak_name = "bf16 sustained (power cap seen)" if power_capped else "bf16 burst (no power cap seen)"
    kernels = {}
    for kind, (cnt, tot) in per_kind.items():
        avg = tot / cnt
        gemm = kind in GEMM_KINDS
        rate = work[kind] / (avg / 1000.0)
        kernels[kind] = {
            "launches_per_step": cnt / prof_steps, "avg_ms": round(avg, 5),
            "share": round(tot / sum(v[1] for v in per_kind.values()), 4),
            "achieved": round(rate / (1e12 if gemm else 1e9), 2),
            "unit": "TFLOP/s" if gemm else "GB/s",
            "frac": round(rate / (1e12 if gemm else 1e9) / (tensor_peak if gemm else peaks["hbm_gbs"]), 4)}
    # dominant kernel: largest total time per step
    dom = max(per_kind, key=lambda k: per_kind[k][1])
    dk = kernels[dom]
    gemm = dk["unit"] == "TFLOP/s"
    traffic = None
    rec = NCU_TRAFFIC.get(dom)
    if rec and rec.get("source_hash") == kernel_source_hash(dom):
        traffic = rec["bytes_per_launch"]
    roofline = {"kernel": dom, "bound": "tensor" if gemm else "hbm", "achieved": dk["achieved"],
                "peak": tensor_peak if gemm else peaks["hbm_gbs"],
                "unit": dk["unit"], "frac": dk["frac"], "traffic": traffic,
                "traffic_source": ("ncu capture of this kernel source (dram read + write bytes per "
                                   "launch), not measured in this run") if traffic else None,
                "peak_source": f"{peaks['source']} ({tensor_peak_name if gemm else 'HBM copy'})"}
    if gemm:
        roofline["frac_of_burst"] = round(dk["achieved"] / peaks["bf16_tflops"], 4)
        roofline["frac_of_sustained"] = round(dk["achieved"] / peaks["bf16_tflops_sustained"], 4)
    gemm_ms = sum(per_kind[k][1] for k in per_kind if k in GEMM_KINDS) / prof_steps
    mom_ms = per_kind.get("momentum", [1, 0.0])[1] / prof_steps

    # ---- the page's update tail after the step (equaliser + sign-aligned decay update
    # on a bf16 + mantissa master weight), timed alone on graph replays: as a separate call
    # on the step's outputs, and with the step-to-tail link (the step also writes the slow
    # rail's sign bits, which the tail reads instead of the fp32 rail); the link's cost in
    # the step is the momentum kernel's extra time in eager steps that write it
    gen = torch.Generator(device=dev).manual_seed(5)
    elems = sum(b.shape[0] * b.shape[1] * b.shape[2] for b in banks)

    def time_tail(links):
        tails = []
        for b, lk in zip(banks, links):
            g_, m_, n_ = b.shape
            nl = m_ if m_ >= n_ else n_
            bits = (torch.randn((g_, m_, n_), device=dev, generator=gen) * 0.05).view(torch.int32)
            tails.append(anvil.Tail(b.out, b.velocity, torch.zeros((g_, nl), dtype=torch.float32, device=dev),
                                    (bits >> 16).to(torch.int16).view(torch.bfloat16).contiguous(),
                                    (bits & 0xFFFF).to(torch.int16).contiguous(),
                                    torch.full((g_,), 0.02, dtype=torch.float32, device=dev), 0.1, 0.95,
                                    tail_link=lk))
        tail_ws = torch.empty(anvil.tail_workspace_bytes([b.shape for b in banks]), dtype=torch.uint8, device=dev)
        with torch.cuda.stream(stream):
            anvil.update_tail(tails, tail_ws, stream=stream)
            g_tail = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_tail, stream=stream):
                anvil.update_tail(tails, tail_ws, stream=stream)
            for _ in range(nwarm):
                g_tail.replay()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(nsteps, 20)
        with torch.cuda.stream(stream):
            t0.record(stream)
            for _ in range(reps):
                g_tail.replay()
            t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / reps

    def tail_entry(ms, bytes_per_elem, note):
        tb = elems * bytes_per_elem
        return {"ms_per_step": ms, "achieved": tb / (ms / 1000.0) / 1e9, "unit": "GB/s",
                "frac": tb / (ms / 1000.0) / 1e9 / peaks["hbm_gbs"], "bytes_per_step": tb, "note": note}

    # algorithmic bytes per element: lane powers read update 2; the apply reads update 2,
    # param and mantissa 2 x 2 and the gate (the fp32 rail 4, or the link's sign words 0.25)
    # and writes param and mantissa 2 x 2
    update_tail = tail_entry(time_tail([None] * len(banks)), 16.0,
                             "3 launches: lane powers (2 B/elem), lane scales, fused equalise + decay (14 B/elem)")
    links = [anvil.alloc_tail_link(b.shape, device=dev) for b in banks]
    for b, lk in zip(banks, links):
        b.tail_link = lk
    with torch.cuda.stream(stream):
        for s in range(2):
            anvil.multi_bank_step(banks, ws, stream=stream)
        torch.cuda.synchronize()
        with anvil.profile(max_records=prof_steps * launches_per_step + 8) as prof_l:
            for s in range(prof_steps):
                for b, gt in zip(banks, pool_d[s % wl.pool]):
                    b.grad = gt
                anvil.multi_bank_step(banks, ws, stream=stream)
    torch.cuda.synchronize()
    mom_link = [t for k, t in prof_l.records if k == "momentum"]
    update_tail_linked = tail_entry(time_tail(links), 12.25,
                                    "3 launches: lane powers (2 B/elem), lane scales, fused equalise + decay gated by the "
                                    "slow-rail sign bits the step wrote into the tail link (10.25 B/elem)")
    update_tail_linked["step_cost_ms"] = statistics.mean(mom_link) - mom_ms
    update_tail_linked["step_cost_note"] = ("the momentum kernel's extra time per step for writing the "
                                            "link's sign bits (eager steps, CUDA events)")
    for b in banks:
        b.tail_link = None

    # ---- the page's Adam step on an lm_head-sized fp32 parameter (768 x 50304)
    cnt = 768 * 50304
    adam_t = [torch.randn(cnt, device=dev, generator=gen) * s_ for s_ in (0.1, 0.01, 0.01)]
    adam_t.append(torch.rand(cnt, device=dev, generator=gen) * 1e-4)
    with torch.cuda.stream(stream):
        for _ in range(nwarm):
            anvil.adam_step(adam_t[0], adam_t[1], adam_t[2], adam_t[3], 0.9, 0.95, 1e-8, 1e-3, 0.0,
                            stream=stream)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(max(nsteps, 20)):
            anvil.adam_step(adam_t[0], adam_t[1], adam_t[2], adam_t[3], 0.9, 0.95, 1e-8, 1e-3, 0.0,
                            stream=stream)
        a1.record(stream)
    torch.cuda.synchronize()
    adam_ms = a0.elapsed_time(a1) / max(nsteps, 20)
    adam_gbs = cnt * 28.0 / (adam_ms / 1000.0) / 1e9
    adam = {"params": cnt, "ms": adam_ms, "achieved": adam_gbs, "unit": "GB/s",
            "frac": adam_gbs / peaks["hbm_gbs"], "bytes_per_param": 28}
    del adam_t

    # ---- end to end: every step copies its gradients in from pinned host memory and
    # its outputs back; the copies of neighbouring steps overlap the current step's
    # compute (two device buffer sets, one upload and one download stream), all inside
    # the timed region.
    host_pool = [[torch.from_numpy(x).pin_memory() for x in p] for p in pool_h]
    gbufs = [[torch.empty_like(x) for x in pool_d[0]] for _ in range(2)]
    outs = [[torch.empty_like(b.out) for b in banks] for _ in range(2)]
    out_h = [torch.empty(b.out.shape, dtype=torch.bfloat16).pin_memory() for b in banks]
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("h2d", "comp", "d2h")}
    main_outs = [b.out for b in banks]
    g_e2e = []
    with torch.cuda.stream(stream):
        for bset in range(2):
            for b, o in zip(banks, outs[bset]):
                b.out = o
            g_e2e.append(capture(gbufs[bset]))
    for b, o in zip(banks, main_outs):
        b.out = o
    torch.cuda.synchronize()

    def e2e_steps(first, count):
        for s in range(first, first + count):
            bset = s & 1
            with torch.cuda.stream(h2d_s):
                if s >= 2:
                    h2d_s.wait_event(ev["comp"][bset])      # step s-2 done reading gbufs[bset]
                for dst, src in zip(gbufs[bset], host_pool[s % wl.pool]):
                    dst.copy_(src, non_blocking=True)
                ev["h2d"][bset].record(h2d_s)
            stream.wait_event(ev["h2d"][bset])
            if s >= 2:
                stream.wait_event(ev["d2h"][bset])          # outs[bset] of step s-2 copied out
            with torch.cuda.stream(stream):
                g_e2e[bset].replay()
            ev["comp"][bset].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev["comp"][bset])
                for dst, o in zip(out_h, outs[bset]):
                    dst.copy_(o, non_blocking=True)
                ev["d2h"][bset].record(d2h_s)

    e2e_steps(0, nwarm)
    torch.cuda.synchronize()
    barrier(world)
    q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    q0.record(h2d_s)
    e2e_steps(nwarm, nsteps)
    d2h_s.wait_event(ev["comp"][(nwarm + nsteps - 1) & 1])
    q1.record(d2h_s)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(q0.elapsed_time(q1) / nsteps, world)
    gbuf = gbufs[0]
    h2d = sum(x.numel() * 4 for x in gbuf)
    d2h = sum(b.out.numel() * 2 for b in banks)
    if not all(torch.isfinite(b.out.float()).all() for b in banks):
        raise RuntimeError("non-finite output")
    if anvil.device_error() != anvil.OK:
        raise RuntimeError("device error word set during the bench")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, secs, cores, picks = oracle_sample(wl, 2, min_seconds=10.0)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"two matrices of each bank ({picks}; {secs:.1f} s of CPU work), "
                         f"mean time per matrix extrapolated to the 66-matrix step"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": nsteps,
            "warmup": nwarm, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(world),
            "tflops_algorithmic": alg / (ms_max / 1000.0) / 1e12 * world,
            "tflops_dense_equivalent": dense / (ms_max / 1000.0) / 1e12 * world,
            "gemm_phase_frac_of_peak": (alg / (gemm_ms / 1000.0) / 1e12) / tensor_peak,
            "momentum_frac_of_hbm": (work["momentum"] / (mom_ms / 1000.0) / 1e9) / peaks["hbm_gbs"],
            "profiled_ms_per_step": prof_ms_step,
            "roofline": roofline, "kernels": kernels, "update_tail": update_tail,
            "update_tail_linked": update_tail_linked, "adam": adam,
            "e2e": {"value": mats * world / (e2e_ms / 1000.0), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": launches_per_step * nsteps,
            "clocks": clocks, "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def run_ncu_case():
    """Two eager (non-graph) steps of the bench workload, one grad draw: a short program for
    ncu captures (four launches per step: momentum, norm_d, normalize, the cascade)."""
    import torch
    from polynomial_matrix_whitening_gb300 import anvil
    dev = torch.device("cuda", 0)
    wl = W.workloads()[WORKLOAD]
    sc = wl.scalars(0)
    banks = [anvil.Bank(torch.from_numpy(wl.grad(j, 0)).to(dev),
                        torch.from_numpy(wl.velocity(j)).to(dev),
                        torch.empty((b.g, b.m, b.n), dtype=torch.bfloat16, device=dev),
                        momentum=sc.momentum, fast_beta=sc.fast_beta, fast_weight=sc.fast_weight,
                        slow_beta=sc.slow_beta) for j, b in enumerate(wl.banks)]
    ws = anvil.alloc_workspace([b.shape for b in banks], device=dev)
    for _ in range(2):
        anvil.multi_bank_step(banks, ws)
    torch.cuda.synchronize()
    if anvil.device_error() != anvil.OK:
        raise RuntimeError("device error word set")
    print("ncu case done")


def run_tail_ncu_case():
    """One step of the bench workload that also writes the step-to-tail link, then the
    update tail on its outputs once without and once with the link: a short program for
    ncu captures of the tail kernels."""
    import torch
    from polynomial_matrix_whitening_gb300 import anvil
    dev = torch.device("cuda", 0)
    wl = W.workloads()[WORKLOAD]
    sc = wl.scalars(0)
    banks = [anvil.Bank(torch.from_numpy(wl.grad(j, 0)).to(dev), torch.from_numpy(wl.velocity(j)).to(dev),
                        torch.empty((b.g, b.m, b.n), dtype=torch.bfloat16, device=dev),
                        momentum=sc.momentum, fast_beta=sc.fast_beta, fast_weight=sc.fast_weight,
                        slow_beta=sc.slow_beta, tail_link=anvil.alloc_tail_link((b.g, b.m, b.n), device=dev))
             for j, b in enumerate(wl.banks)]
    anvil.multi_bank_step(banks, anvil.alloc_workspace([b.shape for b in banks], device=dev))
    gen = torch.Generator(device=dev).manual_seed(5)
    tws = torch.empty(anvil.tail_workspace_bytes([b.shape for b in banks]), dtype=torch.uint8, device=dev)
    for link in (False, True):
        tails = []
        for b in banks:
            g_, m_, n_ = b.shape
            bits = (torch.randn((g_, m_, n_), device=dev, generator=gen) * 0.05).view(torch.int32)
            tails.append(anvil.Tail(b.out, b.velocity, torch.zeros((g_, m_ if m_ >= n_ else n_), device=dev),
                                    (bits >> 16).to(torch.int16).view(torch.bfloat16).contiguous(),
                                    (bits & 0xFFFF).to(torch.int16).contiguous(),
                                    torch.full((g_,), 0.02, device=dev), 0.1, 0.95,
                                    tail_link=b.tail_link if link else None))
        anvil.update_tail(tails, tws)
    torch.cuda.synchronize()
    if anvil.device_error() != anvil.OK:
        raise RuntimeError("device error word set")
    print("tail ncu case done")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["anvil", "reference"], default="anvil")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reference-budget", type=float, default=REFERENCE_BUDGET_S,
                    help="CPU seconds the reference arm's warm-up and timed steps may take")
    ap.add_argument("--ncu-case", action="store_true")
    ap.add_argument("--tail-ncu-case", action="store_true")
    args = ap.parse_args()
    if args.ncu_case:
        run_ncu_case()
        return
    if args.tail_ncu_case:
        run_tail_ncu_case()
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_anvil(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
