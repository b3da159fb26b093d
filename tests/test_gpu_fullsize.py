"""GPU parity on the full-size workloads, every output of the heads checked.

The fp64 matrix-product oracle (``oracle.blas``) computes the definition of
attention over the whole sequence fast enough to compare every row of these
workloads, not a sample:

* causal MHA, 8192 tokens, 8 heads, 4 zigzag shards: every O and lse;
* causal GQA, 32768 tokens, 32/8 heads, 8 zigzag shards (the benched step,
  forward then backward with bf16 gradients, exactly as the bench runs it):
  every O and lse of all 32 query heads; every row of query heads 0-3 and
  28-31 for dQ, and every key of key/value heads 0 and 7 for dK and dV
  (heads are independent, and a key head's gradients need exactly its
  group's query heads); the same outputs of the stepwise forward and of the
  multi-GPU ring emulated on this GPU;
* packed documents, 65536 tokens, 8 contiguous shards that split documents:
  every O and lse;
* causal GQA, 65536 tokens, forward then backward (fp32 gradients): every
  row of query heads 0-3 and 28-31 and every key of KV heads 0 and 7.

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


@pytest.fixture(scope="module")
def gqa32k():
    """The 32K workload's inputs and the oracle's O, lse, dQ (q heads 0-3,
    28-31), dK and dV (kv heads 0, 7), computed once for the tests below."""
    w = WORKLOADS["causal_gqa_t32768_p8_zigzag"]
    x = make_inputs(w, seed=0, with_dout=True)
    kvh = [0, w.hkv - 1]
    rq, rk, rv, _, rl, ro = oracle.blas.attention_bwd(x["q"], x["k"], x["v"], x["dout"],
                                                      causal=True, kv_heads=kvh,
                                                      return_out=True)
    return w, x, kvh, dict(o=ro, lse=rl, dq=rq, dk=rk, dv=rv)


def check_edge_groups(ref, kvh, out=None, lse=None, dq=None, dk=None, dv=None, grad_bf16=False):
    h = EDGE_HEADS
    if out is not None:
        assert max_err(to_np(out[:, h]), ref["o"][:, h]) <= TOL_BF16_O
        assert max_err(to_np(lse[h]), ref["lse"][h]) <= TOL_BF16_LSE
    if dq is None:
        return
    for got, r in ((to_np(dq[:, h]), ref["dq"][:, h]), (to_np(dk[:, kvh]), ref["dk"][:, kvh]),
                   (to_np(dv[:, kvh]), ref["dv"][:, kvh])):
        bound = bf16_output_bound(r, TOL_BF16_O) if grad_bf16 else TOL_BF16_O
        assert np.all(np.abs(got - r) <= bound), max_err(got, r)


def test_causal_gqa_t32768_p8_zigzag_benched_step_every_row_of_edge_groups(gqa32k):
    """The benched step (fused forward, then the backward with bf16 dq, dk,
    dv) against the oracle on q heads 0-3, 28-31 and kv heads 0, 7."""
    w, x, kvh, ref = gqa32k
    q, k, v, out, lse = gpu_forward(w, x)
    do = x["dout"].to(DEV)
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    ra.ringattn_bwd(q, k, v, out, lse, do, None, w.num_shards, w.layout, w.causal, dq, dk, dv)
    assert ra.ringattn_get_status() == 0
    check_edge_groups(ref, kvh, out, lse, dq, dk, dv, grad_bf16=True)
    for t in (out, lse, dq, dk, dv):
        assert bool(torch.isfinite(t).all())


def test_causal_gqa_t32768_p8_zigzag_forward_every_head(gqa32k):
    """The benched shape's forward in full: every O and lse of all 32 query
    heads (the oracle's forward for the heads the fixture's backward does
    not cover)."""
    w, x, kvh, ref = gqa32k
    _, _, _, out, lse = gpu_forward(w, x)
    rest = [h for h in range(w.hq) if h not in EDGE_HEADS]
    ro, rl = oracle.blas.attention_fwd(x["q"], x["k"], x["v"], causal=True, heads=rest)
    assert max_err(to_np(out[:, rest]), ro[:, rest]) <= TOL_BF16_O
    assert max_err(to_np(lse[rest]), rl[rest]) <= TOL_BF16_LSE
    check_edge_groups(ref, kvh, out, lse)


def test_causal_gqa_t32768_p8_zigzag_stepwise_every_row_of_edge_groups(gqa32k):
    """The literal ring form (one launch per ring step, log-sum-exp merges)
    at full size."""
    w, x, kvh, ref = gqa32k
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    out, lse = ra.ringattn_fwd_stepwise(q, k, v, None, w.num_shards, w.layout, w.causal)
    assert ra.ringattn_get_status() == 0
    check_edge_groups(ref, kvh, out, lse)


def test_causal_gqa_t32768_p8_zigzag_multi_gpu_ring_emulated(gqa32k):
    """The multi-GPU ring's schedule with its 8 ranks emulated on this GPU
    (own buffers and streams per rank, device-to-device shard transfers):
    forward and fp32-gradient backward against the oracle."""
    from context_long_sequence_fwd_b300 import ring
    w, x, kvh, ref = gqa32k
    q, k, v, do = (x[n].to(DEV) for n in ("q", "k", "v", "dout"))
    out, lse = ring.emulate_ring_fwd(q, k, v, num_shards=w.num_shards, layout=w.layout,
                                     causal=w.causal)
    dq, dk, dv = ring.emulate_ring_bwd(q, k, v, out, lse, do, num_shards=w.num_shards,
                                       layout=w.layout, causal=w.causal)
    torch.cuda.synchronize()
    assert ra.ringattn_get_status() == 0
    check_edge_groups(ref, kvh, out, lse, dq, dk, dv)


def test_varlen_causal_gqa_t65536_p8_contiguous_every_output():
    """The packed workload in full: every O and lse of all 32 query heads."""
    w = WORKLOADS["varlen_causal_gqa_t65536_p8_contiguous"]
    x = make_inputs(w, seed=0)
    _, _, _, out, lse = gpu_forward(w, x)
    ro, rl = oracle.blas.attention_fwd(x["q"], x["k"], x["v"], causal=True,
                                       cu_seqlens=x["cu_seqlens"])
    assert max_err(to_np(out), ro) <= TOL_BF16_O
    assert max_err(to_np(lse), rl) <= TOL_BF16_LSE


def test_causal_gqa_fwdbwd_t65536_p8_zigzag_every_row_of_edge_groups():
    """The 64K fwd+bwd workload on the head subset its check plan names:
    every row of q heads 0-3 and 28-31 for O, lse and dQ, and every key of
    kv heads 0 and 7 for dK and dV (fp32 gradient outputs: the strict
    2e-2 bound)."""
    w = WORKLOADS["causal_gqa_fwdbwd_t65536_p8_zigzag"]
    x = make_inputs(w, seed=0, with_dout=True)
    q, k, v, out, lse = gpu_forward(w, x)
    do = x["dout"].to(DEV)
    dq, dk, dv = (torch.full(t.shape, float("nan"), device=DEV) for t in (q, k, v))
    ra.ringattn_bwd(q, k, v, out, lse, do, None, w.num_shards, w.layout, w.causal, dq, dk, dv,
                    grad_fp32=True)
    assert ra.ringattn_get_status() == 0
    kvh = [0, w.hkv - 1]
    rq, rk, rv, _, rl, ro = oracle.blas.attention_bwd(x["q"], x["k"], x["v"], x["dout"],
                                                      causal=True, kv_heads=kvh,
                                                      return_out=True)
    check_edge_groups(dict(o=ro, lse=rl, dq=rq, dk=rk, dv=rv), kvh, out, lse, dq, dk, dv)
    for t in (out, lse, dq, dk, dv):
        assert bool(torch.isfinite(t).all())
