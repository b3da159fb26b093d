"""The bench's schedules run end to end on the GPU and print a well-formed
line: the fused path, the literal ring form (one launch per ring step plus
merges) and the multi-GPU ring's per-rank schedule emulated on this GPU, at
the 8K-token workload (the timed numbers themselves are not checked here)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def bench_line(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "2",
                        "--warmup", "3", "--no-cpu-baseline",
                        "--workload", "causal_mha_t8192_p4_zigzag", *args],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("schedule,pass_", [("fused", "fwd"), ("stepwise", "fwd"),
                                            ("ring", "fwd"), ("ring", "fwdbwd")])
def test_bench_schedules(schedule, pass_):
    d = bench_line("--schedule", schedule, "--pass", pass_)
    assert d["status"] == "RA_OK"
    assert d["value"] > 0 and d["e2e"]["value"] > 0
    assert d["config"].get("schedule", "fused") == schedule
    assert d["config"]["pass"] == pass_
    # the launches counted from the library's own trace
    P = d["config"]["num_shards"]
    fwd_launches = d["kernels"]["fwd_tc_bf16_kernel"]["launches"]
    per_step = {"fused": 1, "stepwise": P, "ring": P * P}[schedule]
    assert fwd_launches == 2 * per_step
    assert d["gpu_launches"] >= fwd_launches
