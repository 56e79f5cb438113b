#!/usr/bin/env python3
"""Benchmark of libfattn attn_fwd: attention forward TFLOP/s (bf16, 1x GB300)
and fraction of the dense BF16 tensor-core peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one attn_fwd call over the whole workload (B*H*N query rows,
inputs resident in HBM).  FLOPs = 4*B*H*N^2*d, halved under the causal mask.
The default workload is B=1, H=32, N=16384, d=128, causal, Q/K ~ N(0, 3^2):
its inputs (402 MB) exceed the 126 MB L2, so no flush is needed between
steps; smaller workloads flush L2 before every step (outside the timed
events) and are timed step by step.

Prints one JSON line.  Under torchrun (N > 1) every rank runs the same
workload on its own GPU (independent replicas, weak scaling); the time is the
maximum over ranks and rank 0 prints.  ``--impl reference`` times the fp64
CPU oracle instead (rank 0 only), each step one seeded query row per head.
"""
from __future__ import annotations

import argparse
import csv
import glob
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from tiled_online_softmax_fwd_gb300.inputs import (KV_WORKLOADS, VARIANT_WORKLOADS,  # noqa: E402
                                                   WORKLOADS, digest, make_qkv_kv,
                                                   make_workload)

ALL_WORKLOADS = {**WORKLOADS, **VARIANT_WORKLOADS}

DEFAULT_WORKLOAD = "B1_H32_N16384_d128_causal_sigma3"
METRIC = "attention fwd TFLOP/s (bf16, 1×GB300) and % of dense BF16 tensor peak"
L2_BYTES = 126 * 1024 * 1024
FLUSH_BYTES = 1 << 30
FALLBACK_PEAK_TFLOPS = 1900.0
KERNEL_SOURCES = ["tiled_online_softmax_fwd_gb300/csrc/fattn_fwd_sm103.cu",
                  "tiled_online_softmax_fwd_gb300/csrc/ptx_sm103.cuh"]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["bf16_tflops"]), "measured burst cuBLAS bf16 (MEASURED_PEAKS.json)"
    except Exception:
        return FALLBACK_PEAK_TFLOPS, "fallback 1.9 PFLOP/s bf16 (no MEASURED_PEAKS.json)"


def profiled_traffic(workload: str, key: str = "dram_bytes_per_launch"):
    """DRAM bytes per launch (`key`) from a committed ncu summary of this
    kernel source and workload (null when none matches the current source)."""
    want = kernel_source_hash()
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        groups = []  # a "workload" key starts a new group of bench-key fields
        for line in open(path):
            if line.startswith("bench-key "):
                k, _, v = line[len("bench-key "):].strip().partition("=")
                if k.strip() == "workload":
                    groups.append({})
                if groups:
                    groups[-1][k.strip()] = v.strip()
        for fields in groups:
            if fields.get("workload") == workload and fields.get("kernel_source") == want:
                try:
                    return int(float(fields[key])), os.path.basename(path)
                except (KeyError, ValueError):
                    pass
    return None, None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (read-only)."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        rows = [r for r in csv.reader(io.StringIO(self.out or "")) if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i]
                          and "Not" not in r[5 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, x: float) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def nvtx_range(push: bool, name: str = "attn_fwd timed steps"):
    """Open or close an NVTX range (a no-op where torch has no NVTX)."""
    try:
        if push:
            torch.cuda.nvtx.range_push(name)
        else:
            torch.cuda.nvtx.range_pop()
    except Exception:
        pass


def arm_config(w, world: int, in_digest: str, fp16: bool = False) -> dict:
    """The workload as both arms name it (the GPU arm and the oracle's
    reference arm print the same dictionary)."""
    big = w.io_bytes > L2_BYTES
    return {"workload": w.name + ("_fp16" if fp16 else ""), **w.describe(),
            "parallelism": "replicas" if world > 1 else "single",
            "l2": ("inputs larger than L2 (%d MB)" % (w.io_bytes // 10**6)) if big
                  else "L2 flushed (1 GiB write) before every step, outside the timed events",
            "input_digest": in_digest}


# ------------------------------------------------------------------ CPU oracle
REF_ROWS_PER_HEAD = 16


def oracle_rows_for_steps(w, rows_all, steps, per_step=REF_ROWS_PER_HEAD):
    """per_step seeded rows of every head for each step (cycling through the
    sample), enough rows that every host thread has work."""
    per_head = rows_all.view(w.B * w.H, -1)
    cols = per_head.shape[1]
    return [per_head[:, [(s * per_step + j) % cols for j in range(per_step)]].reshape(-1).clone()
            for s in range(steps)]


def rows_flops(w, rows) -> float:
    i = rows % w.N
    keys = (i + 1).double() if w.causal else torch.full_like(i, w.N).double()
    return float((4.0 * keys * w.d).sum())


def cpu_baseline(w, q, k, v, rows_all, budget_s=15.0):
    """The oracle as it stands on this host's cores, over a bounded sample of
    the workload's rows; returns the same metric (TFLOP/s)."""
    import oracle
    threads = oracle.default_threads()
    qd, kd, vd = (t.to(torch.float64) for t in (q, k, v))
    per_head = rows_all.view(w.B * w.H, -1)
    # Past the checked rows, more seeded rows per head, so that the sample
    # fills the time budget (about 10-30 s of CPU work) on a fast host.
    g = torch.Generator("cpu").manual_seed(20250)
    extra = torch.randint(0, w.N, (w.B * w.H, 8 * per_head.shape[1]), generator=g)
    extra += (torch.arange(w.B * w.H, dtype=torch.int64) * w.N)[:, None]
    per_head = torch.cat([per_head.to(torch.int64), extra], 1)
    total_rows, total_flops, t_total, used = 0, 0.0, 0.0, 0
    col = 0
    while t_total < budget_s and col < per_head.shape[1]:
        take = per_head[:, col:col + 8].reshape(-1)
        col += 8
        t0 = time.perf_counter()
        oracle.attn_fwd(qd, kd, vd, w.scale, w.causal, rows=take.numpy(), threads=threads)
        t_total += time.perf_counter() - t0
        total_rows += take.numel()
        total_flops += rows_flops(w, take)
        used += 1
    # The same oracle on one core, over the first block of rows.
    take = per_head[:, :8].reshape(-1)[:64]
    t0 = time.perf_counter()
    oracle.attn_fwd(qd, kd, vd, w.scale, w.causal, rows=take.numpy(), threads=1)
    single = rows_flops(w, take) / (time.perf_counter() - t0) / 1e12
    return {"value": total_flops / t_total / 1e12, "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "single_core_value": single,
            "sample": "%d query rows (%d seeded rows per head x %d heads, all their keys), %.1f s" %
                      (total_rows, total_rows // (w.B * w.H), w.B * w.H, t_total)}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle
    w = ALL_WORKLOADS[args.workload]
    q, k, v, rows_all = make_workload(w, sample_per_head=1024)
    in_digest = digest(q, k, v)
    qd, kd, vd = (t.to(torch.float64) for t in (q, k, v))
    threads = oracle.default_threads()
    plan = oracle_rows_for_steps(w, rows_all, args.warmup + args.steps)
    for s in range(args.warmup):
        oracle.attn_fwd(qd, kd, vd, w.scale, w.causal, rows=plan[s].numpy(), threads=threads)
    flops = 0.0
    t0 = time.perf_counter()
    for s in range(args.warmup, args.warmup + args.steps):
        oracle.attn_fwd(qd, kd, vd, w.scale, w.causal, rows=plan[s].numpy(), threads=threads)
        flops += rows_flops(w, plan[s])
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = ("each step: %d seeded query rows per head (%d rows, all their keys)"
              % (REF_ROWS_PER_HEAD, REF_ROWS_PER_HEAD * w.B * w.H))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": arm_config(w, world, in_digest),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ row ops
BWD_WORKLOADS = ["bwd_" + n for n in WORKLOADS]

ROWOP_WORKLOADS = {
    "softmax_rows_M32768_N4096_f32": ("softmax_rows", 32768, 4096, torch.float32),
    "softmax_rows_M2048_N65536_f32": ("softmax_rows", 2048, 65536, torch.float32),
    "softmax_rows_M32768_N4096_bf16": ("softmax_rows", 32768, 4096, torch.bfloat16),
    "row_sum_M32768_N4096_f32": ("row_sum", 32768, 4096, torch.float32),
}


def run_rowop(args, world, rank, local):
    """Standalone row softmax / row sum: achieved GB/s of algorithmic traffic
    (read x, write y or the sums; a second read of x for rows too long to keep
    in registers is not counted) against the measured HBM copy bandwidth."""
    import oracle
    from tiled_online_softmax_fwd_gb300 import fattn
    torch.cuda.set_device(local)
    op, M, N, dt = ROWOP_WORKLOADS[args.op]
    g = torch.Generator("cpu").manual_seed(7)
    x = (torch.randn(M, N, generator=g) * 4.0).to(dt)
    dx = x.cuda()
    out = torch.empty_like(dx) if op == "softmax_rows" else torch.empty(M, device=dx.device)
    fn = fattn.softmax_rows if op == "softmax_rows" else fattn.row_sum
    esize = dx.element_size()
    algo_bytes = M * N * esize + (M * N * esize if op == "softmax_rows" else M * 4)
    for _ in range(max(3, args.warmup)):
        fn(dx, out=out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        e0.record()
        for _ in range(args.steps):
            fn(dx, out=out)
        e1.record()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    gbs = algo_bytes / (ms * 1e-3) / 1e9
    try:
        peak = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["hbm_gbs"])
        src = "measured copy (MEASURED_PEAKS.json)"
    except Exception:
        peak, src = 6800.0, "fallback 6.8 TB/s"
    rows = min(M, 256)
    t0 = time.perf_counter()
    (oracle.softmax_rows if op == "softmax_rows" else oracle.row_sum)(x[:rows])
    cpu_s = time.perf_counter() - t0
    cpu_gbs = algo_bytes * rows / M / cpu_s / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": "%s GB/s (HBM-bound, 1xGB300)" % op, "value": gbs, "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if dt == torch.float32 else "bf16", "data": "synthetic",
            "config": {"workload": args.op, "M": M, "N": N,
                       "l2": "inputs larger than L2 (%d MB)" % (M * N * esize // 10**6)},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "peak_source": src, "traffic": None,
                         "algorithmic_bytes_per_launch": algo_bytes},
            "gpu_launches": args.steps, "clocks": clocks.summary(),
            "cpu_baseline": {"value": cpu_gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "%d of %d rows" % (rows, M)}}), flush=True)
    return 0


# ------------------------------------------------------------------ backward
def run_bwd(args, world, rank, local):
    """attn_bwd on one of the forward workloads: TFLOP/s of the method's
    algorithmic work (five products, 10*B*H*N^2*d, halved under the causal
    mask; the kernels recompute S and dP once more, which is not counted)."""
    from tiled_online_softmax_fwd_gb300 import fattn
    torch.cuda.set_device(local)
    w = WORKLOADS[args.op[len("bwd_"):]]
    q, k, v, _ = make_workload(w)
    g = torch.Generator("cpu").manual_seed(77)
    dout = torch.randn(q.shape, generator=g).to(torch.bfloat16).cuda()
    dq_, dk_, dv_ = q.cuda(), k.cuda(), v.cuda()
    o, lse = fattn.attn_fwd(dq_, dk_, dv_, causal=w.causal, scale=w.scale)
    gq, gk, gv = torch.empty_like(dq_), torch.empty_like(dk_), torch.empty_like(dv_)
    ws = torch.empty(w.B * w.H * w.N * 4, dtype=torch.uint8, device=dq_.device)

    def step():
        fattn.attn_bwd(dq_, dk_, dv_, o, lse, dout, causal=w.causal, scale=w.scale, workspace=ws,
                       dq=gq, dk=gk, dv=gv)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    flops = 2.5 * w.flops
    value = flops / (ms * 1e-3) / 1e12
    peak, peak_src = measured_peak()
    if rank == 0:
        print(json.dumps({
            "metric": "attention bwd TFLOP/s (bf16, 1xGB300)", "value": value, "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": args.op, **w.describe()},
            "roofline": {"bound": "tensor", "achieved": value, "peak": peak, "unit": "TFLOP/s",
                         "frac": value / peak, "peak_source": peak_src, "traffic": None,
                         "algorithmic_flops_per_launch": flops,
                         "executed_flops_per_launch": 3.5 * w.flops},
            "gpu_launches": 3 * args.steps, "clocks": clocks.summary()}), flush=True)
    return 0


SDPA_OPS = ["sdpa_" + n for n in sorted(WORKLOADS)]


def run_sdpa(args, world, rank, local):
    """Library context, not part of the product: torch's
    scaled_dot_product_attention (bf16, whatever backend torch picks on this
    GPU) timed on the same inputs as the forward workload, so that the
    forward's figure can be read beside a library number."""
    torch.cuda.set_device(local)
    w = WORKLOADS[args.op[len("sdpa_"):]]
    q, k, v, _ = make_workload(w)
    dq_, dk_, dv_ = q.cuda(), k.cuda(), v.cuda()
    sdpa = torch.nn.functional.scaled_dot_product_attention
    label = "library: torch.nn.functional.scaled_dot_product_attention (torch %s)" % torch.__version__

    def step():
        return sdpa(dq_, dk_, dv_, is_causal=bool(w.causal), scale=w.scale)
    try:
        step()
        torch.cuda.synchronize()
    except Exception as e:  # no kernel for this GPU or shape
        if rank == 0:
            print(json.dumps({"impl": label, "unavailable": str(e).splitlines()[0][:200]}),
                  flush=True)
        return 0
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    value = w.flops / (ms * 1e-3) / 1e12
    peak, peak_src = measured_peak()
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "impl": label, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, **w.describe()},
            "frac_of_peak": value / peak, "peak_source": peak_src,
            "clocks": clocks.summary()}), flush=True)
    return 0


# ------------------------------------------------------------------ decode shapes
def peak_hbm():
    try:
        return (float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["hbm_gbs"]),
                "measured copy (MEASURED_PEAKS.json)")
    except Exception:
        return 6800.0, "fallback 6.8 TB/s"


def run_kv(args, world, rank, local):
    """attn_fwd_kv on a decode-shaped workload (Nq queries per head against Nk
    cached keys): GB/s of algorithmic traffic (K, V, Q read once, O and lse
    written once) against the measured HBM copy bandwidth, and TFLOP/s of the
    visible (query, key) pairs against the bf16 peak."""
    import oracle
    from tiled_online_softmax_fwd_gb300 import fattn
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = KV_WORKLOADS[args.op]
    q, k, v = make_qkv_kv(w.B, w.H, w.Nq, w.Nk, w.d, w.seed, w.sigma_qk)
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    do = torch.empty_like(dq)
    dl = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    need = fattn.kv_workspace_size(w.B, w.H, w.Nq, w.Nk, w.d, w.causal, 0)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    splits = 1 if need == 0 else None  # the library's choice; reported below when known

    def step():
        fattn.attn_fwd_kv(dq, dk, dv, causal=w.causal, scale=w.scale, num_splits=0, workspace=ws,
                          out=do, lse=dl, stream=stream)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    kernel_ms = e0.elapsed_time(e1) / args.steps
    barrier(world)
    status = fattn.device_status()
    ms = max_over_ranks(world, kernel_ms)
    gbs = w.io_bytes / (kernel_ms * 1e-3) / 1e9
    tflops = w.flops / (kernel_ms * 1e-3) / 1e12
    hbm, hbm_src = peak_hbm()
    tc, tc_src = measured_peak()
    bound = "hbm" if gbs / hbm >= tflops / tc else "tensor"
    traffic, traffic_src = profiled_traffic(w.name)
    if need > 0:
        rows = w.B * w.H * w.Nq
        per_split = (w.d * 4 + 8) * rows
        splits = max(2, round(need / per_split))

    # End to end: q, k, v from pinned host memory, o and lse back, all timed.
    e2e = None
    if not args.no_e2e:
        hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
        ho = torch.empty_like(q).pin_memory()
        hl = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32).pin_memory()
        n_e2e = max(3, min(args.steps, 10))
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            step()
            ho.copy_(do, non_blocking=True)
            hl.copy_(dl, non_blocking=True)
            torch.cuda.synchronize()
        e2e_ms = (time.perf_counter() - t0) * 1e3 / n_e2e
        e2e = {"value": w.io_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "ms_per_step": e2e_ms, "steps": n_e2e,
               "h2d_bytes_per_step": (q.numel() + k.numel() + v.numel()) * 2,
               "d2h_bytes_per_step": q.numel() * 2 + w.B * w.H * w.Nq * 4}

    if rank != 0:
        return 0
    # The oracle on this host over whole heads' rows until the budget is spent.
    cpu = None
    if not args.no_cpu_baseline:
        qd, kd, vd = (t.to(torch.float64) for t in (q, k, v))
        threads = oracle.default_threads()
        t_cpu, done_bytes, heads = 0.0, 0.0, 0
        while heads == 0 or (t_cpu < args.cpu_budget and heads < w.B * w.H):
            take = torch.arange(heads * w.Nq, (heads + 1) * w.Nq)
            t1 = time.perf_counter()
            oracle.attn_fwd_kv(qd, kd, vd, w.scale, w.causal, rows=take.numpy(), threads=threads)
            t_cpu += time.perf_counter() - t1
            done_bytes += w.io_bytes / (w.B * w.H)
            heads += 1
        cpu = {"value": done_bytes / t_cpu / 1e9, "unit": "GB/s", "cores": threads,
               "kind": "oracle",
               "sample": "%d of %d heads (all their query rows and keys), %.1f s"
                         % (heads, w.B * w.H, t_cpu)}
    line = {
        "metric": "attention fwd GB/s, decode shape (bf16, 1xGB300)", "value": world * gbs,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, **w.describe(), "splits": splits,
                   "l2": "inputs larger than L2 (%d MB)" % (w.io_bytes // 10**6)},
        "tflops": tflops,
        "roofline": {"bound": bound, "achieved": gbs if bound == "hbm" else tflops,
                     "peak": hbm if bound == "hbm" else tc,
                     "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
                     "frac": gbs / hbm if bound == "hbm" else tflops / tc,
                     "peak_source": hbm_src if bound == "hbm" else tc_src, "traffic": traffic,
                     "traffic_source": traffic_src,
                     "hbm_frac": gbs / hbm, "tensor_frac": tflops / tc,
                     "algorithmic_bytes_per_launch": w.io_bytes,
                     "algorithmic_flops_per_launch": w.flops},
        "gpu_launches": args.steps * (2 if need > 0 else 1),
        "clocks": clocks.summary(), "device_status": status}
    if e2e is not None:
        line["e2e"] = e2e
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
def run_gpu(args, world, rank, local):
    from tiled_online_softmax_fwd_gb300 import fattn
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fattn.load()
    w = ALL_WORKLOADS[args.workload]
    q, k, v, rows_all = make_workload(w, dtype=torch.float16 if args.fp16 else torch.bfloat16,
                                      sample_per_head=1024)
    in_digest = digest(q, k, v)
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    do = torch.empty_like(dq)
    dl = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    big = w.io_bytes > L2_BYTES
    # The flush (a write far larger than L2) also keeps the GPU busy while the
    # host enqueues the step, so that the step's events time the device work
    # and not a host-side gap: 1 GiB takes ~0.17 ms to write.
    flush = None if big else torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    # Key-range split when the library recommends it (few work units per SM;
    # bf16 only).
    splits = 1 if (args.split == "off" or args.fp16) else fattn.split_count(w.B, w.H, w.N, w.d,
                                                                           w.causal, dev)
    ws = None
    if splits > 1:
        ws = torch.empty(fattn.split_workspace_size(w.B, w.H, w.N, w.d, splits), dtype=torch.uint8,
                         device=dev)

    def step():
        if splits > 1:
            fattn.attn_fwd_split(dq, dk, dv, causal=w.causal, scale=w.scale, num_splits=splits,
                                 workspace=ws, out=do, lse=dl, stream=stream)
        elif args.fp16:
            fattn.attn_fwd_fp16(dq, dk, dv, causal=w.causal, scale=w.scale, out=do, lse=dl,
                                stream=stream)
        else:
            fattn.attn_fwd(dq, dk, dv, causal=w.causal, scale=w.scale, out=do, lse=dl,
                           stream=stream)

    for _ in range(args.warmup):
        if flush is not None:
            flush.zero_()
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()

    step_ms = None
    with ClockSampler(local) as clocks:
        # An NVTX range marks the timed steps for a profiler's timeline.
        nvtx_range(True)
        t_wall0 = time.perf_counter()
        if big:
            # One event between consecutive steps: the total gives the value,
            # the gaps give the per-step quantiles.
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
            evs[0].record(stream)
            for i in range(args.steps):
                step()
                evs[i + 1].record(stream)
            torch.cuda.synchronize()
            kernel_ms = evs[0].elapsed_time(evs[-1]) / args.steps
            step_ms = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps))
        else:
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            for a, b in evs:
                flush.zero_()
                a.record(stream)
                step()
                b.record(stream)
            torch.cuda.synchronize()
            step_ms = sorted(a.elapsed_time(b) for a, b in evs)
            kernel_ms = sum(step_ms) / args.steps
        wall_ms = (time.perf_counter() - t_wall0) * 1e3 / args.steps
        nvtx_range(False)
    barrier(world)
    torch.cuda.synchronize()
    status = fattn.device_status()
    ms = max_over_ranks(world, kernel_ms)
    value = world * w.flops / (ms * 1e-3) / 1e12
    achieved = w.flops / (kernel_ms * 1e-3) / 1e12
    v_route = "none" if args.fp16 else fattn.v_conversion_route(w.N, w.d, w.causal)
    prepass = int(v_route == "prepass")

    # End to end through the C ABI with host buffers (pinned), copies timed.
    e2e = None
    if not args.no_e2e and not args.fp16:
        hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
        ho = torch.empty_like(q).pin_memory()
        hl = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()
        n_e2e = max(3, min(args.steps, 20))
        for _ in range(2):
            fattn.attn_fwd_host(hq, hk, hv, ho, hl, dq, dk, dv, do, dl, causal=w.causal,
                                scale=w.scale, stream=stream)
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            fattn.attn_fwd_host(hq, hk, hv, ho, hl, dq, dk, dv, do, dl, causal=w.causal,
                                scale=w.scale, stream=stream)
        e2e_ms = max_over_ranks(world, (time.perf_counter() - t0) * 1e3 / n_e2e)
        barrier(world)
        e2e = {"value": world * w.flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": e2e_ms, "steps": n_e2e,
               "h2d_bytes_per_step": 3 * q.numel() * 2,
               "d2h_bytes_per_step": q.numel() * 2 + w.B * w.H * w.N * 4}

    if rank != 0:
        return 0
    peak, peak_src = measured_peak()
    traffic, traffic_src = profiled_traffic(w.name)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16" if args.fp16 else "bf16", "data": "synthetic",
        "config": arm_config(w, world, in_digest, args.fp16),
        "splits": splits,
        "pct_of_peak": 100.0 * achieved / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_source": peak_src, "traffic": traffic,
                     "traffic_source": traffic_src,
                     "algorithmic_flops_per_launch": w.flops,
                     "algorithmic_bytes_per_launch": w.io_bytes},
        "v_conversion": v_route,
        "gpu_launches": args.steps * (1 + (splits > 1) + prepass),
        "kernel": "fattn %s<%d> (tcgen05/TMA, persistent)%s%s%s" % (
            "fwd_single_kernel" if w.d == 256 else "fwd_kernel", w.d,
            " + combine_kernel, %d key-range splits" % splits if splits > 1 else "",
            " after v_to_f16_kernel (V pre-pass)" if prepass else "",
            "; roofline.achieved uses the whole step" if splits > 1 or prepass else ""),
        "wall_ms_per_step": wall_ms,
        "clocks": clocks.summary(),
        "device_status": status,
    }
    if prepass:
        # The V pre-pass's own DRAM traffic per call (the roofline's traffic
        # is the forward kernel's).
        line["roofline"]["traffic_v_prepass"] = profiled_traffic(
            w.name, "v_prepass_dram_bytes_per_launch")[0]
    if step_ms is not None:
        # Per-step times (L2 flushed before each step, or inputs larger than
        # L2 back to back): quantiles of the step time and the achieved
        # bandwidth of the algorithmic bytes.
        def quantile(f):
            return step_ms[min(len(step_ms) - 1, int(f * len(step_ms)))]
        line["step_quantiles_ms"] = {"p20": quantile(0.2), "p50": quantile(0.5),
                                     "p80": quantile(0.8)}
        line["algorithmic_gbs_p50"] = w.io_bytes / (quantile(0.5) * 1e-3) / 1e9
    if not big:
        # The launch floor under the same timing: one 1-element kernel between
        # the same events after the same L2 flush (median of as many steps).
        x = torch.zeros(1, device=dev)
        floor = []
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            x.add_(1.0)
            b.record(stream)
            torch.cuda.synchronize()
            floor.append(a.elapsed_time(b))
        floor.sort()
        line["us_per_step_p50"] = step_ms[len(step_ms) // 2] * 1e3
        line["launch_floor_us"] = floor[len(floor) // 2] * 1e3
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, q, k, v, rows_all, budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(ALL_WORKLOADS))
    ap.add_argument("--impl", default="libfattn", choices=["libfattn", "reference"])
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--op", default=None,
                    choices=sorted(ROWOP_WORKLOADS) + BWD_WORKLOADS + sorted(KV_WORKLOADS) +
                    SDPA_OPS,
                    help="time a row softmax / row sum, backward or decode-shape workload "
                         "instead, or (sdpa_*) torch's attention on a forward workload as context")
    ap.add_argument("--fp16", action="store_true", help="fp16 inputs through attn_fwd_fp16")
    ap.add_argument("--split", default="auto", choices=["auto", "off"],
                    help="key-range split when the library recommends one (auto) or never")
    ap.add_argument("--v-conversion", default="auto", choices=["auto", "on_chip", "prepass"],
                    help="where bf16 calls round V to fp16 (fattn_set_v_conversion)")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl != "reference":
        from tiled_online_softmax_fwd_gb300 import fattn
        fattn.set_v_conversion(args.v_conversion)
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.op and args.op.startswith("bwd_"):
        return run_bwd(args, world, rank, local)
    if args.op in KV_WORKLOADS:
        return run_kv(args, world, rank, local)
    if args.op in SDPA_OPS:
        return run_sdpa(args, world, rank, local)
    if args.op:
        return run_rowop(args, world, rank, local)
    return run_gpu(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
