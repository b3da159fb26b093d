#!/usr/bin/env python
"""Ring-attention throughput on B300: causal-effective TFLOP/s and % of the
dense BF16 tensor peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--pass P]
    python bench.py --impl reference ...      # the fp64 CPU oracle, timed

A step is one pass of the whole ring-attention hot path over one batch of
seeded synthetic input: the fused forward (planner work list, tile kernel,
in-kernel log-sum-exp merge, epilogue) and then the backward (preprocess,
dQ and dK/dV tile kernels).  The default workload is the causal GQA shape
the 60 % forward target is quoted on: 32 query / 8 key-value heads of
dimension 128, 32768 tokens, 8 zigzag shards.  ``--pass fwd`` times the
forward alone.  Inputs (q, k, v, dO: 670 MB at the default) are larger than
the 126 MB L2, so no flush is needed between steps.  N > 1 GPUs run
independent replicas (one process per GPU, launched by torchrun); the value
is the sum over ranks of the work divided by the slowest rank's time.

Prints one JSON line (rank 0).  With ``--results FILE`` the line is also
appended to FILE, and a configuration already recorded there is printed from
it instead of being run again, so a sweep over workloads that was cut short
resumes where it stopped.
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


def power_capped(clk: dict) -> bool:
    """Whether the power cap held the SM clock down while the step was timed
    (flag seen, median clock under load below 90 % of its maximum).  Reported
    beside the roofline, which is always against the burst peak: the timed
    region is well under the seconds-long loop the sustained figure needs."""
    mhz, top = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    return bool("sw_power_cap" in clk.get("reasons", []) and mhz is not None and top
                and mhz < 0.9 * top)


def workload_config(w, cu, pass_, world, seed) -> dict:
    """The `config` object of the JSON line, the same for both arms."""
    f_step = fwd_flops(w, cu) * (3.5 if pass_ == "fwdbwd" else 1.0)
    elem = 2 if w.dtype == "bf16" else 4
    read_mb = (w.total_tokens * (w.hq + 2 * w.hkv) * w.head_dim * elem
               + (2 * w.total_tokens * w.hq * w.head_dim * elem if pass_ == "fwdbwd" else 0)) / 1e6
    return {"workload": w.name, "total_tokens": w.total_tokens, "hq": w.hq, "hkv": w.hkv,
            "head_dim": w.head_dim, "num_shards": w.num_shards,
            "layout": "zigzag" if w.layout == 1 else "contiguous",
            "causal": w.causal, "varlen_docs": None if cu is None else len(cu) - 1,
            "kv_exchange": "allgather" if w.kv_exchange else "ring",
            "heads_k_stride": w.heads_k_stride,
            "pass": pass_, "flops_per_step": f_step,
            "visible_pairs_per_head": visible_pairs(w, cu),
            "parallelism": f"replicas{world}" if world > 1 else "1gpu",
            "l2": "inputs larger than L2 (%.0f MB read per step), no flush" % read_mb,
            "seed": seed}


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


KERNEL_SOURCES = {"fwd_tc_bf16_kernel": "fwd_tc_bf16.cu", "bwd_dkdv_kernel": "bwd_tc_bf16.cu",
                  "bwd_dq_kernel": "bwd_tc_bf16.cu", "ssd_chunk_scan_kernel": "ssd_cp.cu",
                  "ssd_chunk_scan_tc_kernel": "ssd_chunk_tc.cu",
                  "ssd_correction_kernel": "ssd_cp.cu",
                  "ssd_correction_tc_kernel": "ssd_correction_tc.cu"}


def kernel_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload (profiles/<kernel>_<workload>.md), or None if there is none or
    the kernel's source file has changed since the capture."""
    src = os.path.join(ROOT, "context_long_sequence_fwd_b300", "csrc",
                       KERNEL_SOURCES.get(kernel, ""))
    summ = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not (os.path.isfile(src) and os.path.exists(summ)):
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

def oracle_sample(w, inputs, budget_s: float, seed: int, backward: bool, last=None):
    """Times the fp64 oracle on a bounded sample of the workload and returns
    (flops, seconds, description, threads).  When `last` is a dict, the rows
    and results of the final (timed) call of each kind are left in it, for
    sample_errors.

    The sample is random (head, row) outputs: forward rows (O, lse), and for a
    fwd+bwd pass as many backward rows (dQ, with the row's lse and D).  Each
    output is credited with the algorithmic FLOPs it stands for, per visible
    key: 4 D for a forward row (Q K^T and P V), 6 D for a dQ row (Q K^T, dO V^T
    and dS K).  The key side of the backward (dK, dV) is not sampled: the
    oracle computes it per key only after the row statistics of every query
    that sees the key, which makes one sampled key cost O(T^2)."""
    import oracle
    cu = inputs["cu_seqlens"]
    T = w.total_tokens
    names = ("q", "k", "v", "dout") if backward else ("q", "k", "v")
    for n in names:                   # widen once, outside the timed calls
        if n + "64" not in inputs:
            inputs[n + "64"] = np.ascontiguousarray(inputs[n].float().numpy(), np.float64)
    r = np.random.default_rng(seed)
    bounds = [0, T] if cu is None else [int(x) for x in cu]
    starts = np.zeros(T, np.int64)
    ends = np.zeros(T, np.int64)
    for a, b in zip(bounds[:-1], bounds[1:]):
        starts[a:b] = a
        ends[a:b] = b

    def pick(n):
        hs = r.integers(0, w.hq, n).astype(np.int32)
        is_ = r.integers(0, T, n).astype(np.int32)
        nvis = (is_ + 1 - starts[is_]) if w.causal else (ends[is_] - starts[is_])
        return hs, is_, float(nvis.sum())

    def run_fwd(n):
        hs, is_, vis = pick(n)
        t0 = time.perf_counter()
        res = oracle.fwd_rows(inputs["q64"], inputs["k64"], inputs["v64"], hs, is_,
                              causal=w.causal, cu_seqlens=cu)
        t = time.perf_counter() - t0
        if last is not None:
            last["fwd"] = (hs, is_, res)
        return 4.0 * w.head_dim * vis, t

    def run_bwd(n):
        hs, is_, vis = pick(n)
        t0 = time.perf_counter()
        res = oracle.bwd_rows(inputs["q64"], inputs["k64"], inputs["v64"], inputs["dout64"],
                              hs, is_, causal=w.causal, cu_seqlens=cu)
        t = time.perf_counter() - t0
        if last is not None:
            last["bwd"] = (hs, is_, res)
        return 6.0 * w.head_dim * vis, t

    parts = [("forward rows", run_fwd)] + ([("dQ rows", run_bwd)] if backward else [])
    flops, secs, desc = 0.0, 0.0, []
    for name, fn in parts:
        fn(32)                                        # warm the thread pool
        f0, t0 = fn(128)                              # calibrate
        n = int(min(max(budget_s / len(parts) / max(t0 / 128, 1e-6), 32), 400000))
        f1, t1 = fn(n)
        flops += f1
        secs += t1
        desc.append(f"{n} {name}")
    return flops, secs, ", ".join(desc), oracle.num_threads()


def sample_errors(last, out, lse, dq=None):
    """Largest absolute differences between the step's outputs (torch tensors
    [T, Hq, D] and [Hq, T]) and the oracle's on the rows oracle_sample left in
    `last`: the bench line's own parity check, with the bounds the tests use
    (bf16 gradients: 2e-2 plus half a bf16 ulp of the exact value)."""
    import torch
    errs = {}
    if "fwd" in last:
        hs, is_, (ro, rl) = last["fwd"]
        h, i = torch.from_numpy(hs).long(), torch.from_numpy(is_).long()
        o = out.detach()[i.to(out.device), h.to(out.device)].double().cpu().numpy()
        l = lse.detach()[h.to(lse.device), i.to(lse.device)].double().cpu().numpy()
        errs["rows"] = int(hs.size)
        errs["o"] = float(np.max(np.abs(o - ro))) if hs.size else 0.0
        errs["lse"] = float(np.max(np.abs(l - rl))) if hs.size else 0.0
        errs["within_bounds"] = errs["o"] <= 2e-2 and errs["lse"] <= 1e-3
    if "bwd" in last and dq is not None:
        hs, is_, (rq, _, _) = last["bwd"]
        h, i = torch.from_numpy(hs).long(), torch.from_numpy(is_).long()
        g = dq.detach()[i.to(dq.device), h.to(dq.device)].double().cpu().numpy()
        errs["dq_rows"] = int(hs.size)
        errs["dq"] = float(np.max(np.abs(g - rq))) if hs.size else 0.0
        a = np.abs(rq)
        half_ulp = np.where(a > 0, 2.0 ** (np.floor(np.log2(np.where(a > 0, a, 1.0))) - 8), 0.0)
        bound = 2e-2 + (half_ulp if dq.dtype != torch.float32 else 0.0)
        errs["within_bounds"] = bool(errs.get("within_bounds", True) and
                                     np.all(np.abs(g - rq) <= bound))
    return errs


# ----------------------------------------------------------------- ours

# Algorithmic FLOPs of one launch of each kernel, in units of the forward's
# causal-effective FLOPs (2 matmuls per visible pair).  The backward's five
# matmuls (2.5 forward) are split between its two tile kernels by output: the
# dK/dV kernel owns S, dP, dV and dK; the dQ kernel owns dQ (it recomputes S
# and dP, which is overhead, not algorithmic work).
KERNEL_FWD_UNITS = {"fwd_tc_bf16_kernel": 1.0, "bwd_dkdv_kernel": 2.0, "bwd_dq_kernel": 0.5}


def run_ours(args):
    import torch

    import context_long_sequence_fwd_b300 as ra
    from context_long_sequence_fwd_b300 import ring as ra_ring
    from context_long_sequence_fwd_b300.workloads import WORKLOADS, make_inputs

    world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (B300)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    if w.dtype != "bf16":
        raise SystemExit("the throughput bench runs the bf16 workloads")
    backward = args.pass_ == "fwdbwd"
    x = make_inputs(w, seed=args.seed, with_dout=backward)
    cu = x["cu_seqlens"]
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    out = torch.empty_like(q)
    lse = torch.empty(w.hq, w.total_tokens, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    if backward:
        do = x["dout"].to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(max(ra.bwd_workspace_size(q, k), 16), dtype=torch.uint8, device=dev)

    # The schedule: the fused single-GPU path (the default); the literal ring
    # form, one launch per ring step plus log-sum-exp merges (forward); or the
    # multi-GPU ring's per-rank schedule with all P ranks emulated on this GPU
    # (each rank's own rows, buffers and stream; shard transfers by
    # device-to-device copies), set up once outside the timed region.
    sched = args.schedule
    if sched == "stepwise" and backward:
        raise SystemExit("--schedule stepwise times the forward: use --pass fwd")
    if sched == "ring" and w.kv_exchange != ra.RING:
        raise SystemExit("--schedule ring runs the ring exchange; this workload all-gathers K/V")
    if sched == "stepwise":
        ws_step = torch.empty(ra.fwd_stepwise_workspace_size(q, k, w.heads_k_stride),
                              dtype=torch.uint8, device=dev)

    def fwd_on(b):
        if sched == "stepwise":
            ra.ringattn_fwd_stepwise(b["q"], b["k"], b["v"], cu, w.num_shards, w.layout,
                                     w.causal, b["out"], b["lse"], ws_step, stream,
                                     w.heads_k_stride, w.kv_exchange)
        elif sched == "ring":
            o, l = ra_ring.emulate_ring_fwd(b["q"], b["k"], b["v"], num_shards=w.num_shards,
                                            layout=w.layout, causal=w.causal, cu_seqlens=cu)
            b["out"].copy_(o)
            b["lse"].copy_(l)
        else:
            ra.ringattn_fwd(b["q"], b["k"], b["v"], cu, w.num_shards, w.layout, w.causal,
                            b["out"], b["lse"], stream, w.heads_k_stride, w.kv_exchange)

    def bwd_on(b):
        if sched == "ring":
            g = ra_ring.emulate_ring_bwd(b["q"], b["k"], b["v"], b["out"], b["lse"], b["do"],
                                         num_shards=w.num_shards, layout=w.layout,
                                         causal=w.causal, cu_seqlens=cu)
            for n, t in zip(("dq", "dk", "dv"), g):
                b[n].copy_(t)
        else:
            ra.ringattn_bwd(b["q"], b["k"], b["v"], b["out"], b["lse"], b["do"], cu,
                            w.num_shards, w.layout, w.causal, b["dq"], b["dk"], b["dv"], ws,
                            stream, w.heads_k_stride, kv_exchange=w.kv_exchange)

    main_set = {"q": q, "k": k, "v": v, "out": out, "lse": lse}
    if backward:
        main_set.update(do=do, dq=dq, dk=dk, dv=dv)
    emu = None
    if sched == "ring":
        # steady state of the emulated ring: the ranks already hold their rows
        emu = ra_ring.EmulatedRing(q, k, v, num_shards=w.num_shards, layout=w.layout,
                                   causal=w.causal, cu_seqlens=cu)
        if backward:
            ra.ringattn_fwd(q, k, v, cu, w.num_shards, w.layout, w.causal, out, lse, stream,
                            w.heads_k_stride, w.kv_exchange)
            emu.prepare_bwd(out, lse, do)

    def fwd():
        if emu is not None:
            emu.fwd()
        else:
            fwd_on(main_set)

    def bwd():
        if emu is not None:
            emu.bwd()
        else:
            bwd_on(main_set)

    f_fwd = fwd_flops(w, cu)
    f_step = f_fwd * (3.5 if backward else 1.0)
    for _ in range(args.warmup):
        fwd()
        if backward:
            bwd()
    torch.cuda.synchronize()
    if ra.ringattn_get_status() != 0:
        raise SystemExit("kernel reported an error during warm-up")
    ra.trace_collect()  # drop anything recorded before the timed region

    # The timed region: K steps between two events, nothing else recorded
    # on the stream (at small sizes per-launch events cost a visible share
    # of the step).
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t_start.record(stream)
        for i in range(args.steps):
            fwd()
            if backward:
                bwd()
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    status = ra.ringattn_get_status()
    ms_total = t_start.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_total, world)
    clk = clocks.summary()

    # The same K steps again with per-step and per-kernel CUDA events on the
    # launching stream: the kernel table, the forward/backward split and the
    # roofline's kernel durations come from here.
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    evb = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps if backward else 0)]
    torch.cuda.synchronize()
    ra.trace_enable(True)
    for i in range(args.steps):
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        if backward:
            evb[i][0].record(stream)
            bwd()
            evb[i][1].record(stream)
    torch.cuda.synchronize()
    ra.trace_enable(False)
    kernels = ra.trace_collect()
    status = status or ra.ringattn_get_status()
    fwd_ms = [a.elapsed_time(b) for a, b in ev]
    bwd_ms = [a.elapsed_time(b) for a, b in evb]
    peak_mem = torch.cuda.max_memory_allocated(dev)

    # The memory-bound kernels, against the measured copy bandwidth: the
    # backward preprocess (from the instrumented pass) and the
    # standalone log-sum-exp merge of two bf16 partial results of this
    # workload's size (timed here on its own; the fused forward merges in
    # registers and TMEM, the stepwise forward and multi-GPU callers use it).
    hbm = {}
    T_, H_, D_ = w.total_tokens, w.hq, w.head_dim
    if backward and "bwd_preprocess_kernel" in kernels:
        n, ms = kernels["bwd_preprocess_kernel"]
        nbytes = 2 * T_ * H_ * D_ * 2 + H_ * T_ * 4  # read O, dO (bf16); write D (fp32)
        hbm["bwd_preprocess_kernel"] = {"bytes_per_launch": nbytes, "avg_ms": round(ms / n, 4),
                                        "gbs": round(nbytes / (ms / n * 1e-3) / 1e9, 1)}
    oa, ob = torch.randn_like(out), torch.randn_like(out)
    la = torch.randn(H_, T_, device=dev)
    lb = torch.randn(H_, T_, device=dev)
    for _ in range(3):
        ra.attn_lse_merge(oa, la, ob, lb, stream)
    m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 10
    m0.record(stream)
    for _ in range(reps):
        ra.attn_lse_merge(oa, la, ob, lb, stream)
    m1.record(stream)
    torch.cuda.synchronize()
    mms = m0.elapsed_time(m1) / reps
    nbytes = 3 * T_ * H_ * D_ * 2 + 3 * H_ * T_ * 4  # read o_a, o_b, lse_a, lse_b; write o_a, lse_a
    hbm["lse_merge_kernel"] = {"bytes_per_launch": nbytes, "avg_ms": round(mms, 4),
                               "gbs": round(nbytes / (mms * 1e-3) / 1e9, 1)}
    del oa, ob, la, lb

    # End to end through the public API from pinned host memory: every step
    # copies its inputs in and all of its outputs back.  Two buffer sets and
    # two copy streams pipeline the steps, the way a caller overlaps transfers
    # with compute: step i+1's inputs travel while step i computes, and step
    # i's outputs travel while step i+1 computes.
    h_in = [x[n].pin_memory() for n in (("q", "k", "v", "dout") if backward else ("q", "k", "v"))]
    sets = [main_set]
    sets.append({n: torch.empty_like(t) for n, t in sets[0].items()})
    in_names = ["q", "k", "v", "do"][:len(h_in)]
    out_names = ["out", "lse"] + (["dq", "dk", "dv"] if backward else [])
    h_out = {n: torch.empty(sets[0][n].shape, dtype=sets[0][n].dtype).pin_memory()
             for n in out_names}
    # The forward waits only for q, k, v (dO travels while it runs), and O and
    # lse travel back while the backward runs.
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_in_do = [torch.cuda.Event() for _ in range(2)]
    ev_fwd = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    e2e_steps = max(2, args.steps)

    def e2e_step(i):
        b = sets[i % 2]
        with torch.cuda.stream(cin):
            if i >= 2:
                cin.wait_event(ev_done[i % 2])     # step i-2 has read this set's inputs
            for n, h in zip(in_names[:3], h_in[:3]):
                b[n].copy_(h, non_blocking=True)
            ev_in[i % 2].record(cin)
            if backward:
                b["do"].copy_(h_in[3], non_blocking=True)
                ev_in_do[i % 2].record(cin)
        stream.wait_event(ev_in[i % 2])
        if i >= 2:
            stream.wait_event(ev_out[i % 2])       # step i-2's outputs have left this set
        fwd_on(b)
        ev_fwd[i % 2].record(stream)
        if backward:
            stream.wait_event(ev_in_do[i % 2])
            bwd_on(b)
        ev_done[i % 2].record(stream)
        with torch.cuda.stream(cout):
            cout.wait_event(ev_fwd[i % 2])
            for n in ("out", "lse"):
                h_out[n].copy_(b[n], non_blocking=True)
            if backward:
                cout.wait_event(ev_done[i % 2])
                for n in ("dq", "dk", "dv"):
                    h_out[n].copy_(b[n], non_blocking=True)
            ev_out[i % 2].record(cout)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cin)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(cout)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())
    status = status or ra.ringattn_get_status()

    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        last = {}
        f, t, desc, thr = oracle_sample(w, x, args.cpu_budget, args.seed, backward, last)
        cpu = {"value": round(f / t / 1e12, 6), "unit": "TFLOP/s", "cores": thr,
               "kind": "oracle",
               "sample": f"{desc} of the workload (random head and row), fp64, {t:.1f} s"}
        # the same rows of this run's outputs (after the timed region)
        parity = sample_errors(last, main_set["out"], main_set["lse"],
                               main_set["dq"] if backward else None)

    if rank != 0:
        return
    peaks = load_peaks()
    peak = float(peaks["bf16_tflops"])
    peak_s = float(peaks["bf16_tflops_sustained"])
    ms_step = ms_total / args.steps
    value = world * f_step / (ms_step * 1e-3) / 1e12

    # per-kernel device time over the instrumented pass of K steps (CUDA events
    # on the launch stream)
    ktab = {}
    k_total = sum(ms for _, ms in kernels.values()) or 1.0
    for name, (n, ms) in sorted(kernels.items(), key=lambda kv: -kv[1][1]):
        ent = {"launches": n, "avg_ms": round(ms / n, 4), "share": round(ms / k_total, 4)}
        if name in KERNEL_FWD_UNITS:
            # credited work per step over the kernel's device time per step (its
            # launches per step: 1 fused, one per ring step and rank otherwise)
            ent["tflops"] = round(KERNEL_FWD_UNITS[name] * f_fwd * args.steps / (ms * 1e-3)
                                  / 1e12, 2)
        ktab[name] = ent
    top = max((n for n in ktab if n in KERNEL_FWD_UNITS), key=lambda n: ktab[n]["share"])
    achieved = ktab[top]["tflops"]
    roof = {"bound": "tensor", "kernel": top, "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
            "peak_source": f"{peaks['source']} bf16_tflops (burst)",
            "frac_of_sustained": round(achieved / peak_s, 4),
            "power_capped": power_capped(clk),
            "traffic": kernel_traffic(top, args.workload),
            "flops_per_launch": KERNEL_FWD_UNITS[top] * f_fwd * args.steps / ktab[top]["launches"]}
    fwd_mean = statistics.mean(fwd_ms)
    fwd_tf = f_fwd / (fwd_mean * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q, k, v, dO rounded to bf16)",
        "config": {**workload_config(w, cu, args.pass_, world, args.seed),
                   **({} if sched == "fused" else {"schedule": sched})},
        "fwd": {"ms": round(fwd_mean, 4), "tflops": round(fwd_tf, 2),
                "frac": round(fwd_tf / peak, 4), "frac_of_sustained": round(fwd_tf / peak_s, 4)},
        "roofline": roof,
        "kernels": ktab,
        "cpu_baseline": cpu,
        "parity_sample": parity,
        "e2e": {"value": round(world * f_step / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4),
                "steps": e2e_steps,
                "pipelining": "2 buffer sets; copies on 2 streams overlap the previous "
                              "and next steps' compute; dO travels during the forward, "
                              "O and lse during the backward"},
        "gpu_launches": sum(n for n, _ in kernels.values()),
        "kernel_timing": "per-kernel and per-pass CUDA events over a second run of the same "
                         "K steps after the timed region (none inside it)",
        "hbm_kernels": {**{k: {**v, "frac": round(v["gbs"] / float(peaks["hbm_gbs"]), 4)}
                           for k, v in hbm.items()},
                        "peak_gbs": float(peaks["hbm_gbs"]),
                        "peak_source": peaks["source"] + " hbm_gbs (copy)"},
        "clocks": clk,
        "device": torch.cuda.get_device_name(dev),
        "peak_mem_gb": round(peak_mem / 1e9, 3),
        "status": ra.STATUS.get(status, status),
    }
    if backward:
        bm = statistics.mean(bwd_ms)
        bt = 2.5 * f_fwd / (bm * 1e-3) / 1e12
        line["bwd"] = {"ms": round(bm, 4), "tflops": round(bt, 2), "frac": round(bt / peak, 4),
                       "frac_of_sustained": round(bt / peak_s, 4)}
    emit(line)


# --------------------------------------------- Mamba2 selective scan (CP)

SSD_METRIC = "mamba2 CP selective-scan fwd TFLOP/s at 1 B300"
SSD_BLOCK = 128  # tokens per block of the tensor-core chunk scan


def ssd_flops(T, H, P, N) -> float:
    """The scan's algorithmic flops: per token, head and state entry one
    multiply-add into the state and one into the output."""
    return 4.0 * T * H * P * N


def ssd_tc_flops(T, H, P, N, R) -> float:
    """Tensor-core flops one launch of the chunk scan executes: per block of
    Q tokens, [G | Yoff] = C [B | S0]^T (Q x (Q + P) x N), Ydia = M X and
    S^T += (v o B)^T X (Q x P x Q and N x P x Q), each as three fp16 products
    (hi hi, hi lo, lo hi)."""
    L = T // R
    blocks = R * H * -(-L // SSD_BLOCK)
    Q = SSD_BLOCK
    return blocks * 3 * 2.0 * (Q * (Q + P) * N + Q * P * Q + N * P * Q)


def run_ssd(args):
    import torch

    import context_long_sequence_fwd_b300 as ra
    from context_long_sequence_fwd_b300.workloads import SSD_WORKLOADS, make_ssd_inputs

    world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (B300)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = SSD_WORKLOADS[args.workload]
    inp = make_ssd_inputs(w.total_tokens, w.heads, w.head_dim, w.state_dim, w.groups,
                          args.seed, w.packed, w.doc_lo, w.doc_hi)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    stream = torch.cuda.current_stream(dev)
    y = torch.empty_like(d["x"])
    hT = torch.empty(w.heads, w.head_dim, w.state_dim, device=dev)
    ws = torch.empty(ra.ssd_cp_workspace_size(d["x"], d["B"], w.num_shards), dtype=torch.uint8,
                     device=dev)

    def step(x=d["x"]):
        ra.ssd_cp_fwd(x, d["dt"], d["A"], d["B"], d["C"], d["D"], d["position_ids"],
                      w.num_shards, y, hT, ws, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ra.trace_collect()
    barrier(world)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, world)
    # the same K steps again with per-kernel CUDA events (kernel table, roofline)
    ra.trace_enable(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    ra.trace_enable(False)
    kernels = ra.trace_collect()
    status = ra.ringattn_get_status()
    # End to end: every step's inputs in from pinned host memory and y and the
    # final state back.  Two device buffer sets and two copy streams pipeline
    # the steps the way a caller would: step i+1's inputs travel while step i
    # computes, and step i's outputs travel while step i+1 computes.
    h_in = {k: v.pin_memory() for k, v in inp.items() if v is not None}
    h_y = torch.empty(y.shape).pin_memory()
    h_s = torch.empty(hT.shape).pin_memory()
    sets = [{**{k: d[k] for k in h_in}, "y": y, "hT": hT},
            {**{k: torch.empty_like(d[k]) for k in h_in}, "y": torch.empty_like(y),
             "hT": torch.empty_like(hT)}]
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        b = sets[i % 2]
        with torch.cuda.stream(cin):
            if i >= 2:
                cin.wait_event(ev_done[i % 2])     # step i-2 has read this set's inputs
            for k, v in h_in.items():
                b[k].copy_(v, non_blocking=True)
            ev_in[i % 2].record(cin)
        stream.wait_event(ev_in[i % 2])
        if i >= 2:
            stream.wait_event(ev_out[i % 2])       # step i-2's outputs have left this set
        ra.ssd_cp_fwd(b["x"], b["dt"], b["A"], b["B"], b["C"], b["D"], b.get("position_ids"),
                      w.num_shards, b["y"], b["hT"], ws, stream)
        ev_done[i % 2].record(stream)
        with torch.cuda.stream(cout):
            cout.wait_event(ev_done[i % 2])
            h_y.copy_(b["y"], non_blocking=True)
            h_s.copy_(b["hT"], non_blocking=True)
            ev_out[i % 2].record(cout)

    e2e_steps = max(2, args.steps)
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cin)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(cout)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        heads = max(1, min(w.heads, int(args.cpu_budget * 2)))  # about 0.5 s per head
        t_c = time.perf_counter()
        ry, _ = oracle.ssd_scan(inp["x"][:, :heads], inp["dt"][:, :heads], inp["A"][:heads],
                                inp["B"][:, :1], inp["C"][:, :1], inp["D"][:heads],
                                inp["position_ids"])
        dt_c = time.perf_counter() - t_c
        cpu = {"value": round(ssd_flops(w.total_tokens, heads, w.head_dim, w.state_dim) /
                              dt_c / 1e12, 6),
               "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{heads} of {w.heads} heads over all {w.total_tokens} tokens, fp64, "
                         f"{dt_c:.1f} s"}
        # the sample's heads of group 0 (the timed call reads group 0's B and C
        # for every head) against this run's y, at the tests' 2e-5 relative bound
        g0 = min(heads, w.heads // w.groups)
        ref = np.asarray(ry)[:, :g0]
        got = y[:, :g0].double().cpu().numpy()
        scale = max(1.0, float(np.max(np.abs(ref))))
        rel = float(np.max(np.abs(got - ref))) / scale
        parity = {"heads": g0, "tokens": w.total_tokens, "y_rel": rel,
                  "within_bounds": rel <= 2e-5}
    if rank != 0:
        return
    f = ssd_flops(w.total_tokens, w.heads, w.head_dim, w.state_dim)
    clk = clocks.summary()
    peaks = load_peaks()
    # fp16 products run at the bf16 rate: the measured bf16 burst peak
    peak = float(peaks["bf16_tflops"])
    ktab = {k: {"launches": n, "avg_ms": round(t / n, 4)} for k, (n, t) in kernels.items()}
    scan_kernel = "ssd_chunk_scan_tc_kernel"
    scan_ms = ktab.get(scan_kernel, {}).get("avg_ms", ms)
    f_tc = ssd_tc_flops(w.total_tokens, w.heads, w.head_dim, w.state_dim, w.num_shards)
    achieved = f_tc / (scan_ms * 1e-3) / 1e12
    h2d = sum(v.numel() * v.element_size() for v in h_in.values())
    line = {
        "metric": SSD_METRIC, "value": round(world * f / (ms * 1e-3) / 1e12, 3),
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp16x3/f32",
        "data": "synthetic (seeded; Mamba2 parameter ranges, packed samples)",
        "config": {"workload": w.name, "total_tokens": w.total_tokens, "heads": w.heads,
                   "head_dim": w.head_dim, "state_dim": w.state_dim, "groups": w.groups,
                   "num_shards": w.num_shards, "packed": w.packed,
                   "parallelism": f"replicas{world}" if world > 1 else "1gpu",
                   "l2": "inputs larger than L2 (%.0f MB), no flush" % (h2d / 1e6)},
        "roofline": {"bound": "tensor", "kernel": scan_kernel,
                     "achieved": round(achieved, 3), "peak": round(peak, 1),
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peaks['source']} bf16_tflops (burst; fp16 runs at the "
                                    f"bf16 rate)",
                     "traffic": kernel_traffic(scan_kernel, w.name),
                     "flops_per_launch": f_tc,
                     "recurrence_flops_per_launch": f},
        "kernels": ktab,
        "cpu_baseline": cpu,
        "parity_sample": parity,
        "e2e": {"value": round(world * f / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": h_y.numel() * 4 + h_s.numel() * 4,
                "ms_per_step": round(e2e_ms, 4),
                "steps": e2e_steps,
                "pipelining": "2 buffer sets; copies on 2 streams overlap the previous "
                              "and next steps' compute; dO travels during the forward, "
                              "O and lse during the backward"},
        "gpu_launches": sum(n for n, _ in kernels.values()),
        "kernel_timing": "per-kernel CUDA events over a second run of the same K steps after "
                         "the timed region (none inside it)",
        "clocks": clk,
        "device": torch.cuda.get_device_name(dev),
        "status": ra.STATUS.get(status, status),
    }
    emit(line)


# ------------------------------------------------------------- reference

def run_reference(args):
    """The oracle as it stands, on the host cores, on bounded samples of the
    same workload and pass (the reference arm of the comparison).

    ms_per_step is the measured wall time of one sampled step; the time a
    whole step of the workload would take at the sampled rate is reported
    separately as ms_per_full_step_extrapolated."""
    from context_long_sequence_fwd_b300.workloads import WORKLOADS, make_inputs
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    backward = args.pass_ == "fwdbwd"
    x = make_inputs(w, seed=args.seed, with_dout=backward)
    budget = max(0.5, min(args.cpu_budget, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        oracle_sample(w, x, min(budget, 1.0), args.seed + 1000 + i, backward)
    fl, ts, descs, thr = 0.0, 0.0, [], 1
    for i in range(args.steps):
        f, t, desc, thr = oracle_sample(w, x, budget, args.seed + i, backward)
        fl += f
        ts += t
        descs.append(desc)
    value = fl / ts / 1e12
    f_step = fwd_flops(w, x["cu_seqlens"]) * (3.5 if backward else 1.0)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ts / args.steps * 1e3, 3),
        "ms_per_full_step_extrapolated": round(f_step / (value * 1e12) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) q, k, v, dO rounded to bf16)",
        "config": workload_config(w, x["cu_seqlens"], args.pass_, world, args.seed),
        "sampled": "each step times the oracle on a bounded random sample of the workload's "
                   "rows (see cpu_baseline.sample)",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                         "sample": f"per step: {descs[0]} (random head and row); "
                                   f"{args.steps} steps, {ts:.1f} s"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    emit(line)


# --results FILE: each finished run appends {"run_key": ..., "line": ...} to FILE,
# and a run whose key is already there prints the stored line instead of
# running again, so an interrupted sweep of configurations resumes where it
# stopped (the op keeps no state of its own to checkpoint).
_RESULTS = {"path": None, "key": None}


def run_key(args) -> dict:
    return {"impl": args.impl, "workload": args.workload, "pass": args.pass_,
            "schedule": args.schedule, "gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "seed": args.seed}


def stored_line(path, key):
    if not path or not os.path.exists(path):
        return None
    found = None
    with open(path) as f:
        for raw in f:
            try:
                rec = json.loads(raw)
            except ValueError:
                continue  # a line cut short by an interrupted run
            if isinstance(rec, dict) and rec.get("run_key") == key:
                found = rec.get("line")
    return found


def emit(line):
    """Prints the run's JSON line (and records it with --results)."""
    print(json.dumps(line), flush=True)
    if _RESULTS["path"]:
        path = _RESULTS["path"]
        # a line cut short by an interrupted run stays on a line of its own
        cut = os.path.exists(path) and os.path.getsize(path) > 0
        if cut:
            with open(path, "rb") as f:
                f.seek(-1, os.SEEK_END)
                cut = f.read(1) != b"\n"
        with open(path, "a") as f:
            f.write(("\n" if cut else "") + json.dumps({"run_key": _RESULTS["key"], "line": line})
                    + "\n")


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "fwdbwd"], default="fwdbwd",
                    help="fwd: forward only; fwdbwd: forward then backward (the whole path)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--schedule", choices=["fused", "stepwise", "ring"], default="fused",
                    help="fused single-GPU path; stepwise: one launch per ring step plus "
                         "merges (forward); ring: the multi-GPU ring's per-rank schedule with "
                         "the P ranks emulated on this GPU")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--results", default=None,
                    help="append each finished run to this file; a run already recorded "
                         "there prints its stored line and does not run again")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.results:
        key = run_key(args)
        done = stored_line(args.results, key)
        if done is not None:
            if int(os.environ.get("RANK", "0")) == 0:
                print(json.dumps(done), flush=True)
            return
        # only rank 0 prints, so only rank 0 records
        if int(os.environ.get("RANK", "0")) == 0:
            _RESULTS.update(path=args.results, key=key)
    sys.path.insert(0, ROOT)
    from context_long_sequence_fwd_b300.workloads import SSD_WORKLOADS
    if args.workload in SSD_WORKLOADS:
        if args.impl == "reference":
            raise SystemExit("the SSD workload's reference arm is its cpu_baseline entry")
        run_ssd(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
