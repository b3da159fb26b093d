"""Host-side logic of bench.py, without a GPU: the FLOP accounting and the
multi-process path (replicas: a barrier, the max of the ranks' times, and
rank 0 alone printing), run as world-size-2 gloo ranks on the CPU."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from context_long_sequence_fwd_b300.workloads import WORKLOADS  # noqa: E402


def test_flop_accounting():
    w = WORKLOADS["causal_gqa_t32768_p8_zigzag"]
    # causal: 4 Hq D T^2 / 2 (two matmuls of 2 flops per multiply-add, half the pairs)
    assert bench.fwd_flops(w, None) == 4.0 * 32 * 128 * 32768 ** 2 / 2
    assert bench.visible_pairs(w, None) == 32768 * 32769 // 2
    t = WORKLOADS["tiny_fp32_noncausal_t256"]
    assert bench.fwd_flops(t, None) == 4.0 * 2 * 64 * 256 ** 2
    # packed documents: the sum over documents of L^2
    v = WORKLOADS["varlen_causal_gqa_t65536_p8_contiguous"]
    cu = [0, 1000, 1000, 65536]
    assert bench.fwd_flops(v, cu) == 4.0 * 32 * 128 * (1000 ** 2 + 64536 ** 2) / 2
    assert bench.visible_pairs(v, cu) == 1000 * 1001 // 2 + 64536 * 64537 // 2


def test_ssd_flop_accounting():
    # the recurrence: one multiply-add into the state and one into y per
    # token, head and state entry
    assert bench.ssd_flops(32768, 128, 64, 128) == 4.0 * 32768 * 128 * 64 * 128
    # the chunk scan's executed fp16 products per 128-token block:
    # [G | Yoff] 128 x (128 + 64) x 128, Ydia 128 x 64 x 128, S^T 128 x 64 x 128,
    # three products each for the hi/lo split
    per_block = 3 * 2.0 * (128 * 192 * 128 + 128 * 64 * 128 + 128 * 64 * 128)
    assert bench.ssd_tc_flops(32768, 128, 64, 128, 8) == 8 * 128 * 32 * per_block
    # chunks of 250 tokens: two blocks each, the second one partial
    assert bench.ssd_tc_flops(1000, 4, 64, 128, 4) == 4 * 4 * 2 * per_block


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    # the slowest rank's time is the job's time
    q.put((rank, bench.max_over_ranks(10.0 + rank, world)))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 11.0, 1: 11.0}


def test_reference_arm_under_torchrun_prints_once():
    """Two ranks of the reference arm: rank 0 alone times the oracle and
    prints one JSON line; rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--cpu-budget", "0.5", "--workload", "tiny_fp32_noncausal_t256", "--pass", "fwd"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_ours_refuses_without_gpu():
    """The product arm never falls back to the CPU."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    r = subprocess.run([sys.executable, "bench.py", "--steps", "1", "--warmup", "3"], cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "needs a CUDA device" in (r.stdout + r.stderr)


def test_power_capped_rule():
    """The sustained peak applies only when the cap actually held the clock
    down; a flag seen at full clock (a short forward) keeps the burst peak."""
    cap = ["sw_power_cap"]
    assert bench.power_capped({"sm_mhz": 1530.0, "sm_max_mhz": 2032.0, "reasons": cap})
    assert not bench.power_capped({"sm_mhz": 2028.5, "sm_max_mhz": 2032.0, "reasons": cap})
    assert not bench.power_capped({"sm_mhz": 1530.0, "sm_max_mhz": 2032.0, "reasons": []})
    assert not bench.power_capped({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]})


def test_committed_profiles_parse():
    """Every committed kernel summary the bench reads carries a source digest
    and a DRAM byte count (the digest decides whether the count is used)."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for kernel in bench.KERNEL_SOURCES:
        for name in os.listdir(os.path.join(root, "profiles")):
            if not name.startswith(kernel + "_"):
                continue
            text = open(os.path.join(root, "profiles", name)).read()
            assert "- kernel_source_sha256_16: `" in text, name
            assert "- dram_bytes_per_launch: `" in text, name


def test_results_file_resumes_a_sweep(tmp_path):
    """--results: a run whose configuration is already recorded prints the
    stored line and does not run (so no GPU is needed here); a different
    configuration is not taken for it, and a line cut short by an
    interrupted run is skipped."""
    res = tmp_path / "runs.jsonl"
    args = ["--steps", "2", "--warmup", "3", "--no-cpu-baseline", "--pass", "fwd"]
    key = {"impl": "ours", "workload": bench.DEFAULT_WORKLOAD, "pass": "fwd",
           "schedule": "fused", "gpus": 1, "steps": 2, "warmup": 3, "seed": 0}
    other = dict(key, steps=5)
    with open(res, "w") as f:
        f.write(json.dumps({"run_key": other, "line": {"value": 1.0}}) + "\n")
        f.write(json.dumps({"run_key": key, "line": {"value": 2.0, "metric": "m"}}) + "\n")
        f.write('{"run_key": {"impl": "ours", "workl')  # interrupted
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--results", str(res),
                        *args], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    assert json.loads(r.stdout.strip().splitlines()[-1]) == {"value": 2.0, "metric": "m"}
    assert bench.stored_line(str(res), dict(key, seed=1)) is None
    # a record appended after the cut line stays readable
    bench._RESULTS.update(path=str(res), key=dict(key, seed=1))
    try:
        bench.emit({"value": 3.0})
    finally:
        bench._RESULTS.update(path=None, key=None)
    assert bench.stored_line(str(res), dict(key, seed=1)) == {"value": 3.0}


def test_parity_sample_of_the_bench_line():
    """The bench line's parity sample: the oracle rows the CPU-baseline leg
    computed, compared with the step's outputs at the same (head, row)."""
    import numpy as np
    import torch
    from context_long_sequence_fwd_b300.workloads import make_inputs
    import oracle
    w = WORKLOADS["tiny_fp32_noncausal_t256"]
    x = make_inputs(w, seed=0, with_dout=True)
    last = {}
    bench.oracle_sample(w, x, 0.05, 0, True, last)
    assert set(last) == {"fwd", "bwd"}
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], causal=w.causal)
    rq, _, _, _, _ = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dout"], causal=w.causal)
    out, lse = torch.from_numpy(ro).float(), torch.from_numpy(rl).float()
    dq = torch.from_numpy(rq).to(torch.bfloat16)
    e = bench.sample_errors(last, out, lse, dq)
    assert e["within_bounds"] and e["o"] < 1e-6 and e["lse"] < 1e-5 and e["dq"] < 1e-2
    hs, is_, _ = last["fwd"]
    out[int(is_[0]), int(hs[0]), 0] += 0.5   # a planted error in one sampled output
    e = bench.sample_errors(last, out, lse, dq)
    assert not e["within_bounds"] and abs(e["o"] - 0.5) < 1e-3
    assert np.isfinite(e["dq"])
