"""Writes the golden fixtures of this folder from the fp64 oracle.

    python tests/golden/make_golden.py

Only ``oracle/`` computes the stored values; the inputs come from the seeded
generators (``workloads.make_qkv``), whose bytes are fingerprinted in the
fixture so a change of generator shows up as a failed check rather than as a
silent change of expected values.

The pages print no attention values for a worked example (they give memory
arithmetic only), so every fixture here is a regression freeze of the oracle
on a small case of the definition it follows: exact softmax attention over the
whole sequence, positions reset per packed sample (axolotl "Sequence
Parallelism" page, introduction and "Sample Packing with Sequence
Parallelism").
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from context_long_sequence_fwd_b300.workloads import make_qkv  # noqa: E402

# A 12-token packed sequence of two documents (7 and 5 tokens), 2 query
# heads sharing 1 key/value head, D = 64, fp32, causal; the GPU side runs it
# with 2 zigzag shards (chunks of 3 tokens).
CASES = {
    "causal_varlen_gqa_fp32_t12": dict(T=12, hq=2, hkv=1, d=64, seed=5, causal=True,
                                       cu_seqlens=[0, 7, 12], num_shards=2, layout="zigzag"),
}


def input_digest(tensors) -> str:
    h = hashlib.sha256()
    for t in tensors:
        h.update(np.ascontiguousarray(t.numpy(), np.float32).tobytes())
    return h.hexdigest()


def rows(a):
    return [[float("%.12e" % x) for x in r] for r in np.asarray(a).reshape(-1, a.shape[-1])]


def make(name, c):
    q, k, v, do = make_qkv(c["T"], c["hq"], c["hkv"], c["d"], "fp32", c["seed"], with_dout=True)
    o, lse = oracle.attention_fwd(q, k, v, causal=c["causal"], cu_seqlens=c["cu_seqlens"])
    dq, dk, dv, _, _ = oracle.attention_bwd(q, k, v, do, causal=c["causal"],
                                            cu_seqlens=c["cu_seqlens"])
    return {
        "case": name,
        "source": "fp64 oracle (oracle/attention_fp64.c), written by tests/golden/make_golden.py",
        "inputs": dict(c, dtype="fp32", generator="workloads.make_qkv(T, hq, hkv, d, 'fp32', "
                                                  "seed, with_dout=True)",
                       sha256_q_k_v_dout=input_digest((q, k, v, do))),
        "layouts": {"o": "[T*Hq rows, D]", "lse": "[Hq, T]", "dq": "[T*Hq rows, D]",
                    "dk": "[T*Hkv rows, D]", "dv": "[T*Hkv rows, D]"},
        "o": rows(o), "lse": rows(lse), "dq": rows(dq), "dk": rows(dk), "dv": rows(dv),
    }


def main():
    for name, c in CASES.items():
        path = os.path.join(HERE, name + ".json")
        with open(path, "w") as f:
            json.dump(make(name, c), f, separators=(",", ":"))
            f.write("\n")
        print(path)


if __name__ == "__main__":
    main()
