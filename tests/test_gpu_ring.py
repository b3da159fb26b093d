"""The multi-GPU ring, emulated on one GPU, against the oracle.

Every rank has its own device buffers (its rows of q, k, v, and in the
backward of out, lse and dO), its own stream and its own receive buffers;
the K/V shards (and, in the backward, their dK/dV accumulators) move between
ranks by device-to-device copies ordered with events -- the schedule the
multi-GPU ring runs, with one rank per GPU (aicassindra "tm_sp_math",
"Context parallelism is the axis that is independent"; axolotl "Sequence
Parallelism" page, introduction).  Each step runs ringattn_fwd_rank_step /
ringattn_bwd_rank_step on shard-local buffers.  The gathered results must
match the oracle's attention over the whole sequence.
"""
import numpy as np
import pytest
import torch

import context_long_sequence_fwd_b300 as ra
import oracle
from context_long_sequence_fwd_b300 import ring
from context_long_sequence_fwd_b300.workloads import make_qkv
from tests._util import TOL_BF16_LSE, TOL_BF16_O, max_err, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

CASES = [
    # T, hq, hkv, d, P, layout, causal, cu
    (1024, 4, 2, 128, 2, ra.ZIGZAG, True, None),
    (2048, 8, 2, 128, 4, ra.ZIGZAG, True, None),
    (2048, 4, 2, 128, 8, ra.CONTIGUOUS, True, None),          # ranks that see nothing of later shards
    (1040, 4, 1, 128, 4, ra.ZIGZAG, True, None),              # chunks of 130 rows: ragged tiles
    (2048, 4, 2, 128, 4, ra.CONTIGUOUS, True, [0, 300, 301, 900, 1500, 2048]),  # documents split by shards
    (1536, 6, 2, 128, 3, ra.CONTIGUOUS, False, None),         # non-causal, 3 ranks
    (1024, 4, 4, 64, 2, ra.ZIGZAG, True, [0, 100, 100, 700, 1024]),              # head dim 64
    (512, 2, 1, 128, 1, ra.CONTIGUOUS, True, None),           # a ring of one
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_emulated_ring_forward(case):
    T, hq, hkv, d, P, layout, causal, cu = case
    q, k, v = make_qkv(T, hq, hkv, d, "bf16", seed=41)
    out, lse = ring.emulate_ring_fwd(q.to(DEV), k.to(DEV), v.to(DEV), num_shards=P,
                                     layout=layout, causal=causal, cu_seqlens=cu)
    torch.cuda.synchronize()
    assert ra.ringattn_get_status() == 0
    ro, rl = oracle.attention_fwd(q, k, v, causal=causal, cu_seqlens=cu)
    assert max_err(to_np(out), ro) <= TOL_BF16_O
    assert max_err(to_np(lse), rl) <= TOL_BF16_LSE


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_emulated_ring_backward(case):
    """fp32 gradients (the ring accumulates them across steps in fp32)."""
    T, hq, hkv, d, P, layout, causal, cu = case
    q, k, v, do = make_qkv(T, hq, hkv, d, "bf16", seed=42, with_dout=True)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = ring.emulate_ring_fwd(qd, kd, vd, num_shards=P, layout=layout, causal=causal,
                                     cu_seqlens=cu)
    dq, dk, dv = ring.emulate_ring_bwd(qd, kd, vd, out, lse, dod, num_shards=P, layout=layout,
                                       causal=causal, cu_seqlens=cu)
    torch.cuda.synchronize()
    assert ra.ringattn_get_status() == 0
    rq, rk, rv, _, _ = oracle.attention_bwd(q, k, v, do, causal=causal, cu_seqlens=cu)
    errs = (max_err(to_np(dq), rq), max_err(to_np(dk), rk), max_err(to_np(dv), rv))
    assert max(errs) <= TOL_BF16_O, errs


def test_emulated_ring_matches_fused_step_at_8k():
    """The causal MHA shape at 8192 tokens with 4 zigzag ranks: the ring's
    gathered result against the fused single-GPU forward and backward (both
    compared with the oracle elsewhere), on every output."""
    T, hq, hkv, P = 8192, 8, 8, 4
    q, k, v, do = (t.to(DEV) for t in make_qkv(T, hq, hkv, 128, "bf16", seed=43, with_dout=True))
    out, lse = ring.emulate_ring_fwd(q, k, v, num_shards=P, layout=ra.ZIGZAG, causal=True)
    o2, l2 = ra.ringattn_fwd(q, k, v, None, P, ra.ZIGZAG, True)
    dq, dk, dv = ring.emulate_ring_bwd(q, k, v, out, lse, do, num_shards=P, layout=ra.ZIGZAG,
                                       causal=True)
    g2 = ra.ringattn_bwd(q, k, v, o2, l2, do, None, P, ra.ZIGZAG, True, grad_fp32=True)
    torch.cuda.synchronize()
    assert ra.ringattn_get_status() == 0
    assert max_err(to_np(out), to_np(o2)) <= 1.6e-2
    assert max_err(to_np(lse), to_np(l2)) <= 1e-4
    for a, b in zip((dq, dk, dv), g2):
        assert max_err(to_np(a), to_np(b)) <= 2e-2
