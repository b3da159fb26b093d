#!/usr/bin/env python
"""Ring-attention throughput on B300: causal-effective TFLOP/s and % of the
dense BF16 tensor peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...      # the fp64 CPU oracle, timed

A step is one pass of the ring-attention hot path over one batch of seeded
synthetic input of the named workload (default: causal GQA, 32 query / 8
key-value heads of dimension 128, 32768 tokens, 8 zigzag shards -- the shape
the 60 % target is quoted on).  Forward workloads run the fused forward;
the fwd+bwd workload runs forward then backward.  Inputs (q, k, v: 400 MB at
the default) are larger than the 126 MB L2, so no flush is needed between
steps.  N > 1 GPUs run independent replicas (one process per GPU, launched by
torchrun); the value is the sum over ranks of the work divided by the
slowest rank's time.

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "ring-attn fwd/bwd TFLOP/s (causal-effective) at 1 B300; % of dense BF16 peak"
DEFAULT_WORKLOAD = "causal_gqa_t32768_p8_zigzag"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ------------------------------------------------------------- accounting

def doc_lengths_of(w, cu):
    if cu is None:
        return [w.total_tokens]
    c = [int(x) for x in cu]
    return [b - a for a, b in zip(c[:-1], c[1:])]


def fwd_flops(w, cu) -> float:
    """Causal-effective forward FLOPs: 4 Hq D sum L^2, halved when causal."""
    s = sum(float(L) * L for L in doc_lengths_of(w, cu))
    f = 4.0 * w.hq * w.head_dim * s
    return f / 2 if w.causal else f


def visible_pairs(w, cu) -> int:
    """Exact (query, key) pairs the mask keeps, per head."""
    ls = doc_lengths_of(w, cu)
    return int(sum(L * (L + 1) // 2 for L in ls) if w.causal else sum(L * L for L in ls))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["source"] = "fallback"
    return d


def kernel_traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, if the kernel source is unchanged since the capture."""
    src = os.path.join(ROOT, "context_long_sequence_fwd_b300", "csrc", kernel_file)
    summ = os.path.join(ROOT, "profiles", f"{kernel_file.split('.')[0]}_{workload}.md")
    if not (os.path.exists(src) and os.path.exists(summ)):
        return None
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    vals = {}
    for line in open(summ):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256_16") != digest:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v == "Active"})
        loaded = [r for r in rows if r[2] > 200.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(r[2] for r in rows)}


# ------------------------------------------------------------ distributed

def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------- CPU oracle

def oracle_sample(w, inputs, budget_s: float, seed: int):
    """Times the fp64 oracle on a bounded sample of the workload's rows and
    returns (flops_done, seconds, rows, threads)."""
    import oracle
    cu = inputs["cu_seqlens"]
    T = w.total_tokens
    if "q64" not in inputs:          # widen once, outside the timed calls
        for n in ("q", "k", "v"):
            inputs[n + "64"] = np.ascontiguousarray(inputs[n].float().numpy(), np.float64)
    r = np.random.default_rng(seed)
    bounds = [0, T] if cu is None else [int(x) for x in cu]
    starts = np.zeros(T, np.int64)
    ends = np.zeros(T, np.int64)
    for a, b in zip(bounds[:-1], bounds[1:]):
        starts[a:b] = a
        ends[a:b] = b

    def run(n):
        hs = r.integers(0, w.hq, n).astype(np.int32)
        is_ = r.integers(0, T, n).astype(np.int32)
        nvis = (is_ + 1 - starts[is_]) if w.causal else (ends[is_] - starts[is_])
        t0 = time.perf_counter()
        oracle.fwd_rows(inputs["q64"], inputs["k64"], inputs["v64"], hs, is_,
                        causal=w.causal, cu_seqlens=cu)
        dt = time.perf_counter() - t0
        # QK^T and PV per visible key: 4 D flops (the same convention as the GPU count)
        return 4.0 * w.head_dim * float(nvis.sum()), dt, n

    f0, t0, n0 = run(64)                      # calibrate
    per_row = max(t0 / 64, 1e-6)
    n = int(min(max(budget_s / per_row, 64), 200000))
    f1, t1, n1 = run(n)
    return f1, t1, n1, oracle.num_threads()


# ----------------------------------------------------------------- ours

def run_ours(args):
    import torch

    import context_long_sequence_fwd_b300 as ra
    from context_long_sequence_fwd_b300.workloads import WORKLOADS, make_inputs

    world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (B300)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    if w.dtype != "bf16":
        raise SystemExit("the throughput bench runs the bf16 workloads")
    x = make_inputs(w, seed=args.seed)
    cu = x["cu_seqlens"]
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    out = torch.empty_like(q)
    lse = torch.empty(w.hq, w.total_tokens, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    backward = w.backward
    if backward:
        do = x["dout"].to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(max(ra.bwd_workspace_size(q, k), 16), dtype=torch.uint8, device=dev)

    def fwd():
        ra.ringattn_fwd(q, k, v, cu, w.num_shards, w.layout, w.causal, out, lse, stream,
                        w.heads_k_stride)

    def bwd():
        ra.ringattn_bwd(q, k, v, out, lse, do, cu, w.num_shards, w.layout, w.causal, dq, dk,
                        dv, ws, stream, w.heads_k_stride)

    f_fwd = fwd_flops(w, cu)
    f_step = f_fwd * (3.5 if backward else 1.0)
    for _ in range(args.warmup):
        fwd()
        if backward:
            bwd()
    torch.cuda.synchronize()
    if ra.ringattn_get_status() != 0:
        raise SystemExit("kernel reported an error during warm-up")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    evb = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps if backward else 0)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t_start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            fwd()
            ev[i][1].record(stream)
            if backward:
                evb[i][0].record(stream)
                bwd()
                evb[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    status = ra.ringattn_get_status()
    ms_total = t_start.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_total, world)
    fwd_ms = [a.elapsed_time(b) for a, b in ev]
    bwd_ms = [a.elapsed_time(b) for a, b in evb]
    clk = clocks.summary()

    # end to end through the public API from pinned host memory
    hq_, hk_, hv_ = (x[n].pin_memory() for n in ("q", "k", "v"))
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h_do = x["dout"].pin_memory() if backward else None
    if backward:
        h_dq = torch.empty(dq.shape, dtype=dq.dtype).pin_memory()
        h_dk = torch.empty(dk.shape, dtype=dk.dtype).pin_memory()
        h_dv = torch.empty(dv.shape, dtype=dv.dtype).pin_memory()
    e2e_steps = max(1, min(args.steps, 10))

    def e2e_step():
        q.copy_(hq_, non_blocking=True)
        k.copy_(hk_, non_blocking=True)
        v.copy_(hv_, non_blocking=True)
        if backward:
            do.copy_(h_do, non_blocking=True)
        fwd()
        if backward:
            bwd()
            h_dq.copy_(dq, non_blocking=True)
            h_dk.copy_(dk, non_blocking=True)
            h_dv.copy_(dv, non_blocking=True)
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
    h2d = sum(t.numel() * t.element_size() for t in (hq_, hk_, hv_)) + \
        (h_do.numel() * h_do.element_size() if backward else 0)
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size() + \
        (sum(t.numel() * t.element_size() for t in (h_dq, h_dk, h_dv)) if backward else 0)
    status = status or ra.ringattn_get_status()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        f, t, n, thr = oracle_sample(w, x, args.cpu_budget, args.seed)
        cpu = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
               "sample": f"{n} random (head, row) outputs of the workload, fp64, {t:.1f} s"}

    if rank != 0:
        return
    peaks = load_peaks()
    ms_step = ms_total / args.steps
    value = world * f_step / (ms_step * 1e-3) / 1e12
    fwd_mean = statistics.mean(fwd_ms)
    achieved = f_fwd / (fwd_mean * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    roof = {"bound": "tensor", "kernel": "fwd_tc_bf16_kernel", "achieved": round(achieved, 2),
            "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
            "peak_source": f"{peaks['source']} bf16_tflops (burst)",
            "frac_of_sustained": round(achieved / float(peaks["bf16_tflops_sustained"]), 4),
            "traffic": kernel_traffic("fwd_tc_bf16.cu", args.workload),
            "flops_per_launch": f_fwd}
    launches_per_step = 1 + (0 if not backward else BWD_LAUNCHES)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "total_tokens": w.total_tokens, "hq": w.hq,
                   "hkv": w.hkv, "head_dim": w.head_dim, "num_shards": w.num_shards,
                   "layout": "zigzag" if w.layout == 1 else "contiguous",
                   "causal": w.causal, "varlen_docs": None if cu is None else len(cu) - 1,
                   "pass": "fwd+bwd" if backward else "fwd",
                   "flops_per_step": f_step, "visible_pairs_per_head": visible_pairs(w, cu),
                   "parallelism": f"replicas{world}" if world > 1 else "1gpu",
                   "l2": "inputs larger than L2 (q,k,v %.0f MB), no flush" %
                         (sum(t.numel() * t.element_size() for t in (q, k, v)) / 1e6),
                   "seed": args.seed},
        "pct_of_peak": round(100 * achieved / peak, 2),
        "fwd_ms": round(fwd_mean, 4),
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": round(world * f_step / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "status": ra.STATUS.get(status, status),
    }
    if backward:
        bm = statistics.mean(bwd_ms)
        line["bwd_ms"] = round(bm, 4)
        line["bwd_tflops"] = round(2.5 * f_fwd / (bm * 1e-3) / 1e12, 2)
    print(json.dumps(line), flush=True)


BWD_LAUNCHES = 3  # preprocess, dK/dV(/dQ) tile kernel, dQ convert


# ------------------------------------------------------------- reference

def run_reference(args):
    from context_long_sequence_fwd_b300.workloads import WORKLOADS, make_inputs
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    x = make_inputs(w, seed=args.seed)
    budget = max(0.5, min(args.cpu_budget, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        oracle_sample(w, x, min(budget, 1.0), args.seed + 1000 + i)
    fl, ts, rows, thr = 0.0, 0.0, 0, 1
    for i in range(args.steps):
        f, t, n, thr = oracle_sample(w, x, budget, args.seed + i)
        fl += f
        ts += t
        rows += n
    value = fl / ts / 1e12
    f_step = fwd_flops(w, x["cu_seqlens"])
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(f_step / (value * 1e12) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "total_tokens": w.total_tokens, "hq": w.hq,
                   "hkv": w.hkv, "head_dim": w.head_dim, "num_shards": w.num_shards,
                   "pass": "fwd", "sampled": True},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                         "sample": f"{rows} random (head, row) outputs over {args.steps} steps, "
                                   f"{ts:.1f} s"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    sys.path.insert(0, ROOT)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
