"""GPU parity of the ring-attention backward against the fp64 oracle.

The GPU backward takes the GPU forward's O and lse (as a training step does);
the oracle computes dQ, dK, dV from the definition of attention, with D_i as
sum_j P_ij dP_ij (not via O).  Small cases are compared element by element
(the full-size workloads are in test_gpu_fullsize.py).
"""
import numpy as np
import pytest
import torch

import context_long_sequence_fwd_b300 as ra
import oracle
from context_long_sequence_fwd_b300.workloads import make_qkv
from tests._util import TOL_BF16_O, max_err, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
# fp32 gradients sum up to a few thousand fp32 products of magnitude ~10:
# the accumulated rounding stays well below 1e-4
TOL_FP32_GRAD = 1e-4
TOL_BF16_GRAD = TOL_BF16_O


def run_fwd_bwd(q, k, v, do, cu, P, layout, causal, hks=1, grad_fp32=False, exchange=ra.RING):
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = ra.ringattn_fwd(qd, kd, vd, cu, P, layout, causal, heads_k_stride=hks,
                               kv_exchange=exchange)
    gdt = torch.float32 if grad_fp32 else qd.dtype
    dq, dk, dv = (torch.full(t.shape, float("nan"), dtype=gdt, device=DEV) for t in (qd, kd, vd))
    ra.ringattn_bwd(qd, kd, vd, out, lse, dod, cu, P, layout, causal, dq, dk, dv,
                    heads_k_stride=hks, grad_fp32=grad_fp32, kv_exchange=exchange)
    assert ra.ringattn_get_status() == 0
    return to_np(dq), to_np(dk), to_np(dv)


def bf16_output_bound(ref, tol):
    """tol plus half a bf16 ulp of the exact value: the rounding a bf16 output
    cannot avoid (gradients of magnitude >= 4 have ulps of 1/32 and more)."""
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return tol + np.where(a > 0, 2.0 ** (e - 8), 0.0)


def check_full(q, k, v, do, cu, P, layout, causal, tol, hks=1, grad_fp32=False,
               exchange=ra.RING):
    dq, dk, dv = run_fwd_bwd(q, k, v, do, cu, P, layout, causal, hks, grad_fp32, exchange)
    rq, rk, rv, _, _ = oracle.attention_bwd(q, k, v, do, causal=causal, cu_seqlens=cu)
    errs = (max_err(dq, rq), max_err(dk, rk), max_err(dv, rv))
    if grad_fp32 or q.dtype == torch.float32:
        assert max(errs) <= tol, errs
    else:
        for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
            assert np.all(np.abs(got - ref) <= bf16_output_bound(ref, tol)), errs
    return errs


FP32_CASES = [
    (256, 2, 2, 64, 2, ra.CONTIGUOUS, False, None),       # the tiny fp32 workload's shape
    (300, 4, 2, 64, 3, ra.CONTIGUOUS, True, None),
    (512, 4, 2, 64, 4, ra.ZIGZAG, True, [0, 100, 100, 333, 512]),
    (260, 2, 1, 128, 2, ra.ZIGZAG, True, None),
]


@pytest.mark.parametrize("case", FP32_CASES, ids=[str(i) for i in range(len(FP32_CASES))])
def test_fp32_backward(case):
    T, hq, hkv, d, P, layout, causal, cu = case
    q, k, v, do = make_qkv(T, hq, hkv, d, "fp32", seed=4, with_dout=True)
    check_full(q, k, v, do, cu, P, layout, causal, TOL_FP32_GRAD)


# 44 packed documents of 1 to 97 tokens (seeded draw), several per 128-row tile
MANY_DOCS = [0, 79, 88, 106, 129, 147, 225, 310, 367, 371, 381, 414, 457, 518, 565, 591, 607, 675, 747, 751, 763, 807, 845, 932, 983, 1024, 1066, 1131, 1188, 1205, 1277, 1351, 1444, 1521, 1549, 1581, 1644, 1708, 1776, 1861, 1890, 1982, 1983, 1991, 2048]

BF16_CASES = [
    # T, hq, hkv, P, layout, causal, cu
    (256, 2, 2, 1, ra.CONTIGUOUS, False, None),
    (1024, 2, 2, 2, ra.CONTIGUOUS, True, None),
    (1024, 4, 2, 4, ra.ZIGZAG, True, None),
    (1000, 2, 2, 2, ra.CONTIGUOUS, True, None),         # ragged tiles
    (1040, 4, 1, 4, ra.ZIGZAG, True, None),             # zigzag chunks of 130, G = 4
    (777 * 2, 3, 1, 2, ra.CONTIGUOUS, True, None),      # odd group, ragged tail
    (1536, 8, 2, 3, ra.CONTIGUOUS, False, None),
    (2048, 4, 2, 8, ra.CONTIGUOUS, True, [0, 300, 301, 900, 1500, 2048]),
    (2048, 4, 4, 2, ra.ZIGZAG, False, [0, 128, 640, 641, 2048]),
    (1024, 2, 2, 2, ra.CONTIGUOUS, True, [0, 200, 200, 700, 1024]),
    (2048, 4, 2, 16, ra.ZIGZAG, True, None),             # 32 chunks of 64: half tiles
    (1024, 1, 1, 4, ra.ZIGZAG, True, None),              # a single head
    (2048, 4, 2, 4, ra.CONTIGUOUS, True, MANY_DOCS),     # 44 documents shorter than a tile
    (16, 2, 1, 2, ra.ZIGZAG, True, None),                # 4 chunks of 4 tokens
    (2, 1, 1, 1, ra.CONTIGUOUS, True, None),             # two tokens
    (1024, 16, 2, 4, ra.ZIGZAG, True, None),             # GQA group of 8
    (896, 8, 1, 2, ra.CONTIGUOUS, True, [0, 333, 896]),  # one KV head for 8 query heads
]


@pytest.mark.parametrize("grad_fp32", [True, False], ids=["fp32grad", "bf16grad"])
@pytest.mark.parametrize("case", BF16_CASES, ids=[str(i) for i in range(len(BF16_CASES))])
def test_bf16_backward(case, grad_fp32):
    """bf16 inputs, fp32 accumulation.  With fp32 gradient outputs the strict
    max-abs bound holds; bf16 outputs add their own rounding."""
    T, hq, hkv, P, layout, causal, cu = case
    q, k, v, do = make_qkv(T, hq, hkv, 128, "bf16", seed=12, with_dout=True)
    check_full(q, k, v, do, cu, P, layout, causal, TOL_BF16_GRAD, grad_fp32=grad_fp32)


D64_CASES = [BF16_CASES[i] for i in (0, 1, 2, 4, 5, 7, 9, 12, 13, 14, 15, 16)]


@pytest.mark.parametrize("grad_fp32", [True, False], ids=["fp32grad", "bf16grad"])
@pytest.mark.parametrize("case", D64_CASES, ids=[str(i) for i in range(len(D64_CASES))])
def test_bf16_backward_head_dim_64(case, grad_fp32):
    T, hq, hkv, P, layout, causal, cu = case
    q, k, v, do = make_qkv(T, hq, hkv, 64, "bf16", seed=15, with_dout=True)
    check_full(q, k, v, do, cu, P, layout, causal, TOL_BF16_GRAD, grad_fp32=grad_fp32)


def bf16_ulp(x):
    """One bf16 ulp of |x| (8 significant bits)."""
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 0.0)


def test_bwd_layout_and_stride_invariance():
    """Shard count, layout and heads_k_stride change only the order of the
    sums: the bf16 gradients agree within 3e-2 plus one bf16 ulp (two orders'
    fp32 sums may round to adjacent bf16 values; gradients of magnitude >= 4
    have ulps of 1/32)."""
    T, hq, hkv = 2048, 8, 4
    q, k, v, do = make_qkv(T, hq, hkv, 128, "bf16", seed=6, with_dout=True)
    ref = run_fwd_bwd(q, k, v, do, None, 1, ra.CONTIGUOUS, True)
    for P, layout, hks in [(4, ra.ZIGZAG, 2), (8, ra.CONTIGUOUS, 4)]:
        got = run_fwd_bwd(q, k, v, do, None, P, layout, True, hks)
        for a, b in zip(got, ref):
            a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
            assert np.all(np.abs(a - b) <= 3e-2 + bf16_ulp(b)), max_err(a, b)


def test_bwd_unsupported_is_loud():
    q = torch.zeros(256, 2, 96, dtype=torch.bfloat16, device=DEV)
    lse = torch.zeros(2, 256, device=DEV)
    with pytest.raises(ra.RingAttnError) as e:
        ra.ringattn_bwd(q, q, q, q, lse, q, None, 2, ra.CONTIGUOUS, True)
    assert e.value.code == -3


@pytest.mark.parametrize("case", [BF16_CASES[i] for i in (2, 4, 7, 12)], ids=str)
def test_allgather_backward(case):
    """Backward with the gathered-K/V exchange (varlen_llama3 style)."""
    T, hq, hkv, P, layout, causal, cu = case
    q, k, v, do = make_qkv(T, hq, hkv, 128, "bf16", seed=22, with_dout=True)
    check_full(q, k, v, do, cu, P, layout, causal, TOL_BF16_GRAD, grad_fp32=True,
               exchange=ra.ALLGATHER)


@pytest.mark.parametrize("case", [(2048, 8, 4, 2, None), (2048, 8, 4, 4, None),
                                  (1024, 16, 8, 8, None), (2048, 4, 2, 2, [0, 300, 301, 1500, 2048])],
                         ids=str)
def test_ulysses_backward(case):
    """Ulysses head sharding (all-gather exchange, heads_k_stride = Hkv / P:
    Hkv / P key/value heads per rank, a single one in the second and third
    case): the backward against the oracle."""
    T, hq, hkv, P, cu = case
    q, k, v, do = make_qkv(T, hq, hkv, 128, "bf16", seed=32, with_dout=True)
    check_full(q, k, v, do, cu, P, ra.CONTIGUOUS, True, TOL_BF16_GRAD, hks=hkv // P,
               grad_fp32=True, exchange=ra.ALLGATHER)


@pytest.fixture
def flush_every():
    """Sets the dK/dV flush interval for one test and restores the default."""
    def set_(pairs):
        ra.set_bwd_flush_interval(pairs)
    yield set_
    ra.set_bwd_flush_interval(1024)


FLUSH_CASES = [
    # T, hq, hkv, d, P, layout, causal, cu, flush interval in (query tile, head) pairs
    (2048, 4, 2, 128, 4, ra.ZIGZAG, True, None, 1),        # a flush after every pair
    (2048, 4, 1, 128, 2, ra.CONTIGUOUS, True, None, 3),    # group of 4, interval not a multiple
    (1920, 8, 2, 64, 4, ra.ZIGZAG, True, [0, 700, 701, 1920], 2),   # D = 64, packed documents
    (1024, 2, 2, 128, 2, ra.CONTIGUOUS, False, None, 5),   # non-causal
]


@pytest.mark.parametrize("grad_fp32", [True, False], ids=["fp32grad", "bf16grad"])
@pytest.mark.parametrize("case", FLUSH_CASES, ids=[str(i) for i in range(len(FLUSH_CASES))])
def test_dkdv_flushes_keep_the_result(case, grad_fp32, flush_every):
    """The dK/dV kernel's flushes (TMEM sums moved to fp32 memory every few
    pairs and restarted: into fp32 gradients directly, or into the
    workspace's fp32 sums for bf16 ones) against the oracle, with intervals
    short enough that every key tile flushes many times."""
    T, hq, hkv, d, P, layout, causal, cu, every = case
    flush_every(every)
    q, k, v, do = make_qkv(T, hq, hkv, d, "bf16", seed=41, with_dout=True)
    if not grad_fp32:
        qd, kd = q.to(DEV), k.to(DEV)
        assert ra.bwd_workspace_size(qd, kd) > ra.bwd_workspace_size(qd, kd, grad_fp32=True)
    check_full(q, k, v, do, cu, P, layout, causal, TOL_BF16_GRAD, grad_fp32=grad_fp32)


def test_dkdv_flushes_in_the_ring_steps(flush_every):
    """The multi-GPU ring's per-step backward adds each step into fp32
    gradients; with flushes the partial sums go there too."""
    from context_long_sequence_fwd_b300.ring import emulate_ring_bwd
    flush_every(2)
    T, hq, hkv, P = 2048, 4, 2, 4
    q, k, v, do = make_qkv(T, hq, hkv, 128, "bf16", seed=43, with_dout=True)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = ra.ringattn_fwd(qd, kd, vd, None, P, ra.ZIGZAG, True)
    dq, dk, dv = emulate_ring_bwd(qd, kd, vd, out, lse, dod, num_shards=P, layout=ra.ZIGZAG,
                                  causal=True)
    assert ra.ringattn_get_status() == 0
    rq, rk, rv, _, _ = oracle.attention_bwd(q, k, v, do, causal=True)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert max_err(to_np(got), ref) <= TOL_BF16_GRAD
