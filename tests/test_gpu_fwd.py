"""GPU parity of the ring-attention forward against the fp64 oracle.

Every case runs through the C ABI (libringattn.so) on seeded synthetic
inputs and is compared element by element with the oracle's exact
attention over the whole sequence (or, at full workload sizes, on sampled
rows the oracle computes one by one).  Outputs are pre-filled with NaN so an
element the kernels never write fails the comparison.
"""
import numpy as np
import pytest
import torch

import context_long_sequence_fwd_b300 as ra
import oracle
from context_long_sequence_fwd_b300.workloads import (WORKLOADS, cu_seqlens_from_lengths,
                                                      doc_lengths, make_inputs, make_qkv)
from tests._util import (TOL_BF16_LSE, TOL_BF16_O, TOL_FP32, max_err, nan_like, sample_rows,
                         to_np)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_fwd(q, k, v, cu, P, layout, causal, stepwise=False, hks=1, exchange=ra.RING):
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    out = nan_like(qd)
    lse = torch.full((q.shape[1], q.shape[0]), float("nan"), device=DEV)
    if stepwise:
        ra.ringattn_fwd_stepwise(qd, kd, vd, cu, P, layout, causal, out, lse, heads_k_stride=hks,
                                 kv_exchange=exchange)
    else:
        ra.ringattn_fwd(qd, kd, vd, cu, P, layout, causal, out, lse, heads_k_stride=hks,
                        kv_exchange=exchange)
    assert ra.ringattn_get_status() == 0
    return to_np(out), to_np(lse)


def check_full(q, k, v, cu, P, layout, causal, tol_o, tol_l, stepwise=False, hks=1,
               exchange=ra.RING):
    o, l = run_fwd(q, k, v, cu, P, layout, causal, stepwise, hks, exchange)
    ro, rl = oracle.attention_fwd(q, k, v, causal=causal, cu_seqlens=cu)
    eo, el = max_err(o, ro), max_err(l, rl)
    assert eo <= tol_o and el <= tol_l, (eo, el)
    return eo, el


# ------------------------------------------------------------------ fp32

@pytest.mark.parametrize("stepwise", [False, True])
def test_tiny_fp32_noncausal_workload(stepwise):
    """T=256, 2 heads, D=64, P=2 contiguous, non-causal, seed 0: <= 1e-5."""
    w = WORKLOADS["tiny_fp32_noncausal_t256"]
    x = make_inputs(w, seed=0)
    check_full(x["q"], x["k"], x["v"], None, w.num_shards, w.layout, w.causal,
               TOL_FP32, TOL_FP32, stepwise)


@pytest.mark.parametrize("case", [
    (300, 4, 2, 64, 3, ra.CONTIGUOUS, True, None),
    (520, 2, 1, 128, 2, ra.ZIGZAG, True, None),
    (400, 3, 3, 64, 2, ra.CONTIGUOUS, False, [0, 37, 38, 200, 400]),
    (512, 4, 2, 64, 4, ra.ZIGZAG, True, [0, 100, 100, 333, 512]),
])
@pytest.mark.parametrize("stepwise", [False, True])
def test_fp32_paths(case, stepwise):
    T, hq, hkv, d, P, layout, causal, cu = case
    q, k, v = make_qkv(T, hq, hkv, d, "fp32", seed=3)
    check_full(q, k, v, cu, P, layout, causal, TOL_FP32, TOL_FP32, stepwise)


# ------------------------------------------------------------------ bf16

# 44 packed documents of 1 to 97 tokens (seeded draw), several per 128-row tile
MANY_DOCS = [0, 79, 88, 106, 129, 147, 225, 310, 367, 371, 381, 414, 457, 518, 565, 591, 607, 675, 747, 751, 763, 807, 845, 932, 983, 1024, 1066, 1131, 1188, 1205, 1277, 1351, 1444, 1521, 1549, 1581, 1644, 1708, 1776, 1861, 1890, 1982, 1983, 1991, 2048]

BF16_CASES = [
    # T, hq, hkv, P, layout, causal, cu
    (256, 2, 2, 1, ra.CONTIGUOUS, False, None),         # one tile pair, no mask
    (1024, 2, 2, 2, ra.CONTIGUOUS, True, None),         # causal, MHA row pairs
    (1024, 4, 2, 4, ra.ZIGZAG, True, None),             # GQA head pairs, zigzag
    (1000, 2, 2, 2, ra.CONTIGUOUS, True, None),         # chunks of 500: ragged tiles
    (1040, 4, 1, 4, ra.ZIGZAG, True, None),             # zigzag chunks of 130
    (777 * 2, 3, 1, 2, ra.CONTIGUOUS, True, None),      # odd group size, ragged tail
    (1536, 8, 2, 3, ra.CONTIGUOUS, False, None),        # non-causal, 3 shards
    (2048, 4, 2, 8, ra.CONTIGUOUS, True, [0, 300, 301, 900, 1500, 2048]),   # varlen
    (2048, 4, 4, 2, ra.ZIGZAG, False, [0, 128, 640, 641, 2048]),            # varlen non-causal
    (1024, 2, 2, 2, ra.CONTIGUOUS, True, [0, 200, 200, 700, 1024]),         # empty document
    (2048, 4, 2, 16, ra.ZIGZAG, True, None),             # 32 chunks of 64: half tiles
    (1024, 1, 1, 4, ra.ZIGZAG, True, None),              # a single head
    (2048, 4, 2, 4, ra.CONTIGUOUS, True, MANY_DOCS),     # 44 documents shorter than a tile
    (16, 2, 1, 2, ra.ZIGZAG, True, None),                # 4 chunks of 4 tokens
    (2, 1, 1, 1, ra.CONTIGUOUS, True, None),             # two tokens
    (1024, 16, 2, 4, ra.ZIGZAG, True, None),             # GQA group of 8
    (896, 8, 1, 2, ra.CONTIGUOUS, True, [0, 333, 896]),  # one KV head for 8 query heads
]


@pytest.mark.parametrize("case", BF16_CASES, ids=[str(i) for i in range(len(BF16_CASES))])
@pytest.mark.parametrize("stepwise", [False, True])
def test_bf16_small_cases(case, stepwise):
    T, hq, hkv, P, layout, causal, cu = case
    q, k, v = make_qkv(T, hq, hkv, 128, "bf16", seed=11)
    check_full(q, k, v, cu, P, layout, causal, TOL_BF16_O, TOL_BF16_LSE, stepwise)


# head dimension 64: causal, zigzag, GQA (groups of 2, 3, 4 and 8), packed
# documents (an empty one, many short ones), ragged tiles and tiny inputs
D64_CASES = [BF16_CASES[i] for i in (0, 1, 2, 4, 5, 7, 8, 9, 12, 13, 14, 15, 16)]


@pytest.mark.parametrize("case", D64_CASES, ids=[str(i) for i in range(len(D64_CASES))])
@pytest.mark.parametrize("stepwise", [False, True])
def test_bf16_head_dim_64(case, stepwise):
    T, hq, hkv, P, layout, causal, cu = case
    q, k, v = make_qkv(T, hq, hkv, 64, "bf16", seed=13)
    check_full(q, k, v, cu, P, layout, causal, TOL_BF16_O, TOL_BF16_LSE, stepwise)


def test_bf16_head_dim_64_allgather():
    T, hq, hkv, P, layout, causal, cu = BF16_CASES[7]
    q, k, v = make_qkv(T, hq, hkv, 64, "bf16", seed=14)
    check_full(q, k, v, cu, P, layout, causal, TOL_BF16_O, TOL_BF16_LSE, False, 2,
               exchange=ra.ALLGATHER)


def test_bf16_large_scores():
    """Scores far from zero (std ~ 8) exercise the deferred rescaling."""
    q, k, v = make_qkv(1024, 2, 2, 128, "fp32", seed=5)
    q = (q * 8.0).to(torch.bfloat16)
    k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    check_full(q, k, v, None, 2, ra.ZIGZAG, True, TOL_BF16_O, TOL_BF16_LSE)


def test_layout_and_stride_invariance():
    """P, layout and heads_k_stride change the schedule, not the result."""
    T, hq, hkv = 2048, 8, 4
    q, k, v = make_qkv(T, hq, hkv, 128, "bf16", seed=2)
    ref_o, ref_l = run_fwd(q, k, v, None, 1, ra.CONTIGUOUS, True)
    for P, layout, hks in [(2, ra.CONTIGUOUS, 1), (4, ra.ZIGZAG, 2), (8, ra.ZIGZAG, 4),
                           (8, ra.CONTIGUOUS, 1)]:
        o, l = run_fwd(q, k, v, None, P, layout, True, hks=hks)
        # only the accumulation order differs: O agrees to a bf16 ulp or two
        assert max_err(o, ref_o) <= 1.6e-2 and max_err(l, ref_l) <= 1e-4


def test_fused_matches_stepwise():
    T = 2048
    q, k, v = make_qkv(T, 4, 2, 128, "bf16", seed=9)
    cu = [0, 513, 514, 1700, 2048]
    o1, l1 = run_fwd(q, k, v, cu, 4, ra.CONTIGUOUS, True)
    o2, l2 = run_fwd(q, k, v, cu, 4, ra.CONTIGUOUS, True, stepwise=True)
    assert max_err(o1, o2) <= 1.6e-2 and max_err(l1, l2) <= 1e-4


def test_empty_input_is_noop():
    q = torch.empty(0, 2, 128, dtype=torch.bfloat16, device=DEV)
    k = torch.empty(0, 2, 128, dtype=torch.bfloat16, device=DEV)
    out, lse = ra.ringattn_fwd(q, k, k, None, 2, ra.ZIGZAG, True)
    assert out.numel() == 0 and lse.numel() == 0
    assert ra.ringattn_get_status() == 0


def test_unsupported_is_loud():
    q = torch.zeros(256, 2, 96, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ra.RingAttnError) as e:
        ra.ringattn_fwd(q, q, q, None, 2, ra.CONTIGUOUS, True)
    assert e.value.code == -3
    q = torch.zeros(250, 2, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ra.RingAttnError) as e:
        ra.ringattn_fwd(q, q, q, None, 4, ra.CONTIGUOUS, True)
    assert e.value.code == -2


# ------------------------------------------------- full-size workloads

def sampled_check(name, n_rows, seed=0):
    w = WORKLOADS[name]
    x = make_inputs(w, seed=seed)
    cu = x["cu_seqlens"]
    o, l = run_fwd(x["q"], x["k"], x["v"], cu, w.num_shards, w.layout, w.causal,
                   hks=w.heads_k_stride, exchange=w.kv_exchange)
    # rows at shard and zigzag-chunk boundaries, the ends, plus random rows
    C = w.total_tokens // (2 * w.num_shards)
    edges = sorted({0, 1, 127, 128, w.total_tokens - 1} |
                   {c * C for c in range(1, 2 * w.num_shards)} |
                   {c * C - 1 for c in range(1, 2 * w.num_shards)})
    if cu is not None:
        edges += [int(c) for c in cu[1:-1]] + [int(c) - 1 for c in cu[1:-1]]
    hs, is_ = sample_rows(w.total_tokens, w.hq, n_rows, seed + 100, edges[:24])
    ro, rl = oracle.fwd_rows(x["q"], x["k"], x["v"], hs, is_, causal=w.causal, cu_seqlens=cu)
    eo = max_err(o[is_, hs], ro)
    el = max_err(l[hs, is_], rl)
    assert eo <= TOL_BF16_O and el <= TOL_BF16_LSE, (eo, el)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))


def test_causal_gqa_t32768_p8_zigzag():
    sampled_check("causal_gqa_t32768_p8_zigzag", 512)


def test_varlen_causal_gqa_t65536_p8_contiguous():
    sampled_check("varlen_causal_gqa_t65536_p8_contiguous", 384)


def test_concurrent_launches_reuse_work_counters():
    """140 fused forwards on two streams at once (more launches than the
    library's 64 work-counter slots): every result equals the first one bit
    for bit -- each item is computed by exactly one CTA, whichever claims it."""
    T, hq, hkv, P = 2048, 4, 2, 4
    q, k, v = (t.to(DEV) for t in make_qkv(T, hq, hkv, 128, "bf16", seed=9))
    ref_o, ref_l = ra.ringattn_fwd(q, k, v, None, P, ra.ZIGZAG, True)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    results = []
    for i in range(140):
        st = streams[i % 2]
        with torch.cuda.stream(st):
            o = torch.empty_like(q)
            l = torch.empty(hq, T, device=DEV)
            ra.ringattn_fwd(q, k, v, None, P, ra.ZIGZAG, True, o, l, stream=st)
            results.append((o, l))
    torch.cuda.synchronize()
    assert ra.ringattn_get_status() == 0
    for o, l in results:
        assert torch.equal(o, ref_o) and torch.equal(l, ref_l)


@pytest.mark.parametrize("case", [BF16_CASES[i] for i in (2, 4, 7, 9, 12)], ids=str)
@pytest.mark.parametrize("stepwise", [False, True])
def test_allgather_exchange(case, stepwise):
    """varlen_llama3-style exchange: gathered K/V in token order, with two
    key/value heads per pass where the heads allow it."""
    T, hq, hkv, P, layout, causal, cu = case
    q, k, v = make_qkv(T, hq, hkv, 128, "bf16", seed=21)
    hks = 2 if hkv % 2 == 0 else 1
    check_full(q, k, v, cu, P, layout, causal, TOL_BF16_O, TOL_BF16_LSE, stepwise, hks,
               exchange=ra.ALLGATHER)


def test_varlen_causal_gqa_t65536_p8_contiguous_allgather():
    sampled_check("varlen_causal_gqa_t65536_p8_contiguous_allgather", 384)


ULYSSES_CASES = [
    # T, hq, hkv, P, cu: each of P ranks owns Hkv / P key/value heads
    (2048, 8, 4, 2, None),                     # two key/value heads per rank
    (2048, 8, 4, 4, None),                     # a single key/value head per rank
    (1024, 16, 8, 8, None),                    # one per rank, GQA group of 2
    (2048, 4, 2, 2, [0, 300, 301, 1500, 2048]),  # packed documents
]


@pytest.mark.parametrize("case", ULYSSES_CASES, ids=str)
@pytest.mark.parametrize("stepwise", [False, True])
def test_ulysses_head_partition(case, stepwise):
    """DeepSpeed-Ulysses (clusterbid "Sequence Parallelism: GPU Optimization
    Guide 2026") shards heads instead of tokens: each of P ranks attends over
    the whole sequence for Hkv / P key/value heads and their query heads.  On
    one GPU that is the all-gather exchange with heads_k_stride = Hkv / P,
    one pass per rank's head group; compared with the oracle."""
    T, hq, hkv, P, cu = case
    q, k, v = make_qkv(T, hq, hkv, 128, "bf16", seed=31)
    check_full(q, k, v, cu, P, ra.CONTIGUOUS, True, TOL_BF16_O, TOL_BF16_LSE, stepwise,
               hks=hkv // P, exchange=ra.ALLGATHER)


def test_bounded_wait_runs_out_and_is_reported():
    """The kernels' failure path, without a fault: a wait on a barrier that
    nothing arrives at gives up after its limit (about 1 s), the status word
    reports RA_ERR_TIMEOUT once, and the context still computes correctly."""
    import time
    assert ra.ringattn_get_status() == 0
    t0 = time.perf_counter()
    ra.selftest_wait_timeout()
    status = ra.ringattn_get_status()
    elapsed = time.perf_counter() - t0
    assert status == -5, status  # RA_ERR_TIMEOUT
    assert 0.5 < elapsed < 30.0, elapsed
    assert ra.ringattn_get_status() == 0  # read once, then cleared
    q, k, v = make_qkv(512, 2, 1, 128, "bf16", seed=21)
    check_full(q, k, v, None, 2, ra.ZIGZAG, True, TOL_BF16_O, TOL_BF16_LSE, False)
