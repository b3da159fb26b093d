"""GPU parity on the full-size workloads, every output of the heads checked.

The fp64 matrix-product oracle (``oracle.blas``) computes the definition of
attention over the whole sequence fast enough to compare every row of these
workloads, not a sample:

* causal MHA, 8192 tokens, 8 heads, 4 zigzag shards: every O and lse;
* causal GQA, 32768 tokens, 32/8 heads, 8 zigzag shards (the benched step,
  forward then backward with bf16 gradients, exactly as the bench runs it):
  every row of query heads 0-3 and 28-31 for O, lse and dQ, and every key of
  key/value heads 0 and 7 for dK and dV (heads are independent, and a key
  head's gradients need exactly its group's query heads);
* packed documents, 65536 tokens, 8 contiguous shards that split documents:
  every row of query heads 0-3 and 28-31.

The ring schedule reaches the whole-sequence result by re-ordering the sum
(axolotl "Sequence Parallelism" page, introduction: results aggregated
through a ring), so each output is compared with the oracle element by
element within the workloads' bounds.
"""
import numpy as np
import pytest
import torch

import context_long_sequence_fwd_b300 as ra
import oracle
from context_long_sequence_fwd_b300.workloads import WORKLOADS, make_inputs
from tests._util import TOL_BF16_LSE, TOL_BF16_O, max_err, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
EDGE_HEADS = [0, 1, 2, 3, 28, 29, 30, 31]


def bf16_output_bound(ref, tol):
    """tol plus half a bf16 ulp of the exact value: the rounding a bf16 output
    cannot avoid (gradients of magnitude >= 4 have ulps of 1/32 and more)."""
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return tol + np.where(a > 0, 2.0 ** (e - 8), 0.0)


def gpu_forward(w, x):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.hq, w.total_tokens), float("nan"), device=DEV)
    ra.ringattn_fwd(q, k, v, x["cu_seqlens"], w.num_shards, w.layout, w.causal, out, lse,
                    heads_k_stride=w.heads_k_stride, kv_exchange=w.kv_exchange)
    assert ra.ringattn_get_status() == 0
    return q, k, v, out, lse


def test_causal_mha_t8192_p4_zigzag_every_output():
    w = WORKLOADS["causal_mha_t8192_p4_zigzag"]
    x = make_inputs(w, seed=0)
    _, _, _, out, lse = gpu_forward(w, x)
    ro, rl = oracle.blas.attention_fwd(x["q"], x["k"], x["v"], causal=True)
    assert max_err(to_np(out), ro) <= TOL_BF16_O
    assert max_err(to_np(lse), rl) <= TOL_BF16_LSE


def test_causal_gqa_t32768_p8_zigzag_benched_step_every_row_of_edge_groups():
    """The benched step (fused forward, then the backward with bf16 dq, dk,
    dv) against the oracle on q heads 0-3, 28-31 and kv heads 0, 7."""
    w = WORKLOADS["causal_gqa_t32768_p8_zigzag"]
    x = make_inputs(w, seed=0, with_dout=True)
    q, k, v, out, lse = gpu_forward(w, x)
    do = x["dout"].to(DEV)
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    ra.ringattn_bwd(q, k, v, out, lse, do, None, w.num_shards, w.layout, w.causal, dq, dk, dv)
    assert ra.ringattn_get_status() == 0
    kvh = [0, w.hkv - 1]
    rq, rk, rv, _, rl, ro = oracle.blas.attention_bwd(x["q"], x["k"], x["v"], x["dout"],
                                                      causal=True, kv_heads=kvh,
                                                      return_out=True)
    h = EDGE_HEADS
    assert max_err(to_np(out[:, h]), ro[:, h]) <= TOL_BF16_O
    assert max_err(to_np(lse[h]), rl[h]) <= TOL_BF16_LSE
    for got, ref in ((to_np(dq[:, h]), rq[:, h]), (to_np(dk[:, kvh]), rk[:, kvh]),
                     (to_np(dv[:, kvh]), rv[:, kvh])):
        assert np.all(np.abs(got - ref) <= bf16_output_bound(ref, TOL_BF16_O)), max_err(got, ref)
    for t in (out, lse, dq, dk, dv):
        assert bool(torch.isfinite(t).all())


def test_varlen_causal_gqa_t65536_p8_contiguous_every_row_of_edge_groups():
    w = WORKLOADS["varlen_causal_gqa_t65536_p8_contiguous"]
    x = make_inputs(w, seed=0)
    _, _, _, out, lse = gpu_forward(w, x)
    ro, rl = oracle.blas.attention_fwd(x["q"], x["k"], x["v"], causal=True,
                                       cu_seqlens=x["cu_seqlens"], heads=EDGE_HEADS)
    assert max_err(to_np(out[:, EDGE_HEADS]), ro[:, EDGE_HEADS]) <= TOL_BF16_O
    assert max_err(to_np(lse[EDGE_HEADS]), rl[EDGE_HEADS]) <= TOL_BF16_LSE
    assert bool(torch.isfinite(out).all()) and bool(torch.isfinite(lse).all())
