"""The stepwise forward that allocates nothing.

Callers such as an allocator or memory-pool callback, or a host runtime that
only hands out input and output buffers, cannot call cudaMalloc where they
run attention.  ringattn_fwd_stepwise_noalloc serves them from a fixed
library-owned scratch array.  This file checks, through the C ABI, that two
calls in a row give the same result as the workspace-taking
ringattn_fwd_stepwise (within the parity tolerances the other tests use),
that the result matches the fp64 oracle, and that a problem too large for
the array is refused before any launch.  It is
named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import context_long_sequence_fwd_b300 as ra
from context_long_sequence_fwd_b300.workloads import make_qkv
from tests._util import TOL_BF16_LSE, TOL_BF16_O, TOL_FP32, max_err, nan_like, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SCRATCH_BYTES = 32 << 20  # RA_NOALLOC_SCRATCH_BYTES in include/ringattn.h


def noalloc_fn():
    lib = ra.library()
    fn = lib.ringattn_fwd_stepwise_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.POINTER(ctypes.c_int32), ra.ra_dims, ctypes.c_int, ctypes.c_int,
                   ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def call_noalloc(q, k, v, cu, P, layout, causal):
    out = nan_like(q)
    lse = torch.full((q.shape[1], q.shape[0]), float("nan"), device=DEV)
    cu_arr = None if cu is None else np.ascontiguousarray(cu, dtype=np.int32)
    cu_p = None if cu_arr is None else cu_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    dims = ra.make_dims(q, k, 0 if cu_arr is None else cu_arr.size - 1)
    stream = ctypes.c_void_p(int(torch.cuda.current_stream().cuda_stream))
    code = noalloc_fn()(q.data_ptr(), k.data_ptr(), v.data_ptr(), cu_p, dims, P, layout,
                        int(causal), out.data_ptr(), lse.data_ptr(), stream)
    assert code == 0, ra.STATUS.get(code, code)
    return out, lse


CASES = [
    # T, hq, hkv, D, dtype, P, layout, causal, cu
    (2048, 4, 2, 128, "bf16", 4, ra.ZIGZAG, True, None),
    (1000, 2, 2, 128, "bf16", 2, ra.CONTIGUOUS, True, [0, 300, 301, 1000]),
    (256, 2, 2, 64, "fp32", 2, ra.CONTIGUOUS, False, None),
]


def test_two_calls_match_the_workspace_entry_point():
    for (T, hq, hkv, d, dt, P, layout, causal, cu) in CASES:
        q, k, v = (t.to(DEV) for t in make_qkv(T, hq, hkv, d, dt, seed=T))
        ref_o, ref_l = ra.ringattn_fwd_stepwise(q, k, v, cu, P, layout, causal)
        first = call_noalloc(q, k, v, cu, P, layout, causal)
        second = call_noalloc(q, k, v, cu, P, layout, causal)
        assert ra.ringattn_get_status() == 0
        tol_o, tol_l = (TOL_FP32, TOL_FP32) if dt == "fp32" else (TOL_BF16_O, TOL_BF16_LSE)
        for o, l in (first, second):
            assert max_err(to_np(o), to_np(ref_o)) <= tol_o
            assert max_err(to_np(l), to_np(ref_l)) <= tol_l


def test_result_matches_the_oracle():
    """The same cases against the fp64 oracle's whole-sequence attention."""
    import oracle
    for (T, hq, hkv, d, dt, P, layout, causal, cu) in CASES:
        qc, kc, vc = make_qkv(T, hq, hkv, d, dt, seed=T)
        o, l = call_noalloc(qc.to(DEV), kc.to(DEV), vc.to(DEV), cu, P, layout, causal)
        assert ra.ringattn_get_status() == 0
        ro, rl = oracle.attention_fwd(qc, kc, vc, causal=causal, cu_seqlens=cu)
        tol_o, tol_l = (TOL_FP32, TOL_FP32) if dt == "fp32" else (TOL_BF16_O, TOL_BF16_LSE)
        assert max_err(to_np(o), ro) <= tol_o and max_err(to_np(l), rl) <= tol_l


def test_oversized_problem_is_refused():
    # fp32 partials alone: 2 * T * Hq * D * 4 bytes > 32 MiB
    T, hq = 16384, 4
    q = torch.zeros(T, hq, 128, dtype=torch.bfloat16, device=DEV)
    out = torch.zeros_like(q)
    lse = torch.zeros(hq, T, device=DEV)
    dims = ra.make_dims(q, q)
    stream = ctypes.c_void_p(int(torch.cuda.current_stream().cuda_stream))
    code = noalloc_fn()(q.data_ptr(), q.data_ptr(), q.data_ptr(), None, dims, 2,
                        ra.CONTIGUOUS, 1, out.data_ptr(), lse.data_ptr(), stream)
    assert code == -6  # RA_ERR_WORKSPACE
    assert torch.count_nonzero(out).item() == 0
