"""B300-native ring attention: Python binding of ``libringattn.so``.

Argument marshalling only.  Every step of the computation runs in the CUDA
library (``csrc/``), reached through its C ABI (``include/ringattn.h``);
torch tensors are only the owners of device memory and ``torch.cuda``
streams the ordering.  If the library has not been built the import of a
compute function raises: there is no CPU fallback.

Entry points (same names as the C ABI):
    ringattn_fwd, ringattn_fwd_stepwise, ringattn_bwd, attn_lse_merge,
    ringattn_fwd_rank_step / ringattn_bwd_rank_step (one ring step of one rank
    of a multi-GPU ring, on shard-local buffers; ``ring.py`` drives them),
    ringattn_get_status, plan_fwd / plan_bwd (host-only work-list
    introspection), trace_enable / trace_collect (per-kernel device time),
    ssd_cp_fwd (context-parallel Mamba2 selective scan).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

CONTIGUOUS = 0
ZIGZAG = 1
RING = 0        # ring_attn_func batch_ring: K/V shards visited in ring order
ALLGATHER = 1   # ring_attn_func varlen_llama3: gathered K/V in token order
RA_BF16 = 0
RA_FP32 = 1

STATUS = {
    0: "RA_OK", -1: "RA_ERR_INVALID_ARG", -2: "RA_ERR_NOT_DIVISIBLE",
    -3: "RA_ERR_UNSUPPORTED", -4: "RA_ERR_CUDA", -5: "RA_ERR_TIMEOUT",
    -6: "RA_ERR_WORKSPACE", -7: "RA_ERR_BOUNDS",
}
PLAN_ITEM_FIELDS = 16
PLAN_SEG_FIELDS = 4
ITEM_COLUMNS = ("q0_a", "q0_b", "qlen_a", "qlen_b", "head_a", "head_b", "seg_begin",
                "seg_count", "rank", "cost", "mask_lo_a", "mask_lo_b", "mask_hi_a",
                "mask_hi_b", "pass", "part")
SEG_COLUMNS = ("k0", "k1", "step", "src")
PLAN_BWD_ITEM_FIELDS = 8
BWD_ITEM_COLUMNS = ("k0", "klen", "kv_head", "src", "seg_begin", "seg_count", "cost", "pad")
BWD_SEG_COLUMNS = ("q0", "q1", "step", "rank")

_HERE = os.path.dirname(os.path.abspath(__file__))
# RINGATTN_DEBUG=1 selects the bounds-checking build (libringattn_debug.so,
# `python -m context_long_sequence_fwd_b300.build --debug`)
DEBUG = os.environ.get("RINGATTN_DEBUG", "0") not in ("", "0")
LIB_PATH = os.path.join(_HERE, "libringattn_debug.so" if DEBUG else "libringattn.so")
_lib = None


class RingAttnError(RuntimeError):
    def __init__(self, func: str, code: int):
        self.code = code
        super().__init__(f"{func} failed: {STATUS.get(code, code)}")


class ra_dims(ctypes.Structure):
    _fields_ = [("total_tokens", ctypes.c_int), ("num_seqs", ctypes.c_int),
                ("hq", ctypes.c_int), ("hkv", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("dtype", ctypes.c_int), ("heads_k_stride", ctypes.c_int),
                ("grad_fp32", ctypes.c_int), ("kv_exchange", ctypes.c_int)]


class ssd_dims(ctypes.Structure):
    _fields_ = [("total_tokens", ctypes.c_int), ("heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("state_dim", ctypes.c_int),
                ("groups", ctypes.c_int)]


class ra_trace_entry(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_char * 40), ("launches", ctypes.c_int),
                ("total_ms", ctypes.c_double)]


_vp = ctypes.c_void_p
_i32p = ctypes.POINTER(ctypes.c_int32)
_ip = ctypes.POINTER(ctypes.c_int)


def library():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m context_long_sequence_fwd_b300.build"
                + (" --debug" if DEBUG else "") + "` (nvcc, sm_103a)")
        lib = ctypes.CDLL(LIB_PATH)
        lib.ringattn_fwd.argtypes = [_vp, _vp, _vp, _i32p, ra_dims, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, _vp, _vp, _vp]
        lib.ringattn_fwd_stepwise.argtypes = [_vp, _vp, _vp, _i32p, ra_dims, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, _vp, _vp, _vp,
                                              ctypes.c_size_t, _vp]
        lib.ringattn_fwd_stepwise_workspace_size.argtypes = [ra_dims]
        lib.ringattn_fwd_stepwise_workspace_size.restype = ctypes.c_size_t
        lib.ringattn_bwd_workspace_size.argtypes = [ra_dims]
        lib.ringattn_bwd_workspace_size.restype = ctypes.c_size_t
        lib.ringattn_set_bwd_flush_interval.argtypes = [ctypes.c_int]
        lib.ringattn_set_bwd_flush_interval.restype = ctypes.c_int
        lib.ringattn_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32p, ra_dims, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, _vp,
                                     ctypes.c_size_t, _vp]
        lib.attn_lse_merge.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, _vp]
        lib.ringattn_get_status.argtypes = [_vp]
        lib.ringattn_selftest_wait_timeout.argtypes = [_vp]
        lib.ringattn_status_string.argtypes = [ctypes.c_int]
        lib.ringattn_status_string.restype = ctypes.c_char_p
        lib.ringattn_version.restype = ctypes.c_int
        lib.ringattn_debug_report.argtypes = [_vp, ctypes.POINTER(ctypes.c_longlong),
                                              ctypes.POINTER(ctypes.c_longlong)]
        lib.ringattn_debug_report.restype = ctypes.c_int
        lib.ringattn_plan_fwd.argtypes = [_i32p, ra_dims, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, _i32p, ctypes.c_int, _i32p, ctypes.c_int,
                                          _ip, _ip]
        lib.ringattn_plan_bwd.argtypes = lib.ringattn_plan_fwd.argtypes
        lib.ringattn_plan_fwd_fused.argtypes = [_i32p, ra_dims, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int,
                                                _i32p, ctypes.c_int, _ip, _ip]
        lib.ringattn_fwd_rank_workspace_size.argtypes = [ra_dims, ctypes.c_int]
        lib.ringattn_fwd_rank_workspace_size.restype = ctypes.c_size_t
        lib.ringattn_fwd_rank_step.argtypes = [_vp, _vp, _vp, _i32p, ra_dims, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, _vp, _vp, _vp, _vp, _vp,
                                               ctypes.c_size_t, _vp]
        lib.ringattn_bwd_rank_workspace_size.argtypes = [ra_dims, ctypes.c_int]
        lib.ringattn_bwd_rank_workspace_size.restype = ctypes.c_size_t
        lib.ringattn_bwd_rank_step.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32p, ra_dims,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, _vp,
                                               ctypes.c_size_t, _vp]
        lib.ssd_cp_workspace_size.argtypes = [ssd_dims, ctypes.c_int]
        lib.ssd_cp_workspace_size.restype = ctypes.c_size_t
        lib.ssd_cp_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, ssd_dims, ctypes.c_int,
                                   _vp, _vp, _vp, ctypes.c_size_t, _vp]
        lib.ssd_cp_fwd.restype = ctypes.c_int
        lib.ringattn_trace_enable.argtypes = [ctypes.c_int]
        lib.ringattn_trace_collect.argtypes = [ctypes.POINTER(ra_trace_entry), ctypes.c_int, _ip]
        for fn in ("ringattn_fwd", "ringattn_fwd_stepwise", "ringattn_bwd", "attn_lse_merge",
                   "ringattn_fwd_rank_step", "ringattn_bwd_rank_step",
                   "ringattn_get_status", "ringattn_selftest_wait_timeout",
                   "ringattn_plan_fwd", "ringattn_plan_bwd", "ringattn_plan_fwd_fused",
                   "ringattn_trace_enable", "ringattn_trace_collect"):
            getattr(lib, fn).restype = ctypes.c_int
        _lib = lib
    return _lib


def _check(func: str, code: int):
    if code != 0:
        raise RingAttnError(func, code)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return RA_BF16
    if t.dtype == torch.float32:
        return RA_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


def _cu_host(cu_seqlens):
    """cu_seqlens as a host int32 array (the library copies what it needs)."""
    if cu_seqlens is None:
        return None, 0, None
    if hasattr(cu_seqlens, "detach"):
        arr = cu_seqlens.detach().to("cpu").numpy()
    else:
        arr = np.asarray(cu_seqlens)
    arr = np.ascontiguousarray(arr, dtype=np.int32)
    return arr.ctypes.data_as(_i32p), arr.size - 1, arr


def make_dims(q, k, num_seqs=0, heads_k_stride=1, grad_fp32=False, kv_exchange=RING) -> ra_dims:
    T, hq, d = q.shape
    return ra_dims(T, num_seqs, hq, k.shape[1], d, _dtype_code(q), heads_k_stride,
                   int(bool(grad_fp32)), int(kv_exchange))


def _need(t, name, shape=None, dtype=None):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")


def _check_qkv(q, k, v):
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n)
    if k.shape != v.shape or q.shape[0] != k.shape[0] or q.shape[2] != k.shape[2]:
        raise ValueError("q [T,Hq,D], k and v [T,Hkv,D] expected")
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share a dtype")


def ringattn_fwd(q, k, v, cu_seqlens=None, num_shards=1, shard_layout=CONTIGUOUS, causal=True,
                 out=None, lse=None, stream=None, heads_k_stride=1, kv_exchange=RING):
    """Fused ring-attention forward; returns (out [T,Hq,D], lse fp32 [Hq,T])."""
    import torch
    _check_qkv(q, k, v)
    T, hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(hq, T, dtype=torch.float32, device=q.device)
    _need(out, "out", q.shape, q.dtype)
    _need(lse, "lse", (hq, T), torch.float32)
    cu_p, nseq, _keep = _cu_host(cu_seqlens)
    dims = make_dims(q, k, nseq, heads_k_stride, kv_exchange=kv_exchange)
    _check("ringattn_fwd", library().ringattn_fwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), cu_p, dims, int(num_shards),
        int(shard_layout), int(bool(causal)), out.data_ptr(), lse.data_ptr(), _stream(stream)))
    return out, lse


def fwd_stepwise_workspace_size(q, k, heads_k_stride=1) -> int:
    return int(library().ringattn_fwd_stepwise_workspace_size(make_dims(q, k, 0, heads_k_stride)))


def ringattn_fwd_stepwise(q, k, v, cu_seqlens=None, num_shards=1, shard_layout=CONTIGUOUS,
                          causal=True, out=None, lse=None, workspace=None, stream=None,
                          heads_k_stride=1, kv_exchange=RING):
    """Ring forward as one launch per ring step plus a log-sum-exp merge."""
    import torch
    _check_qkv(q, k, v)
    T, hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(hq, T, dtype=torch.float32, device=q.device)
    _need(out, "out", q.shape, q.dtype)
    _need(lse, "lse", (hq, T), torch.float32)
    need = fwd_stepwise_workspace_size(q, k, heads_k_stride)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    cu_p, nseq, _keep = _cu_host(cu_seqlens)
    dims = make_dims(q, k, nseq, heads_k_stride, kv_exchange=kv_exchange)
    _check("ringattn_fwd_stepwise", library().ringattn_fwd_stepwise(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), cu_p, dims, int(num_shards), int(shard_layout),
        int(bool(causal)), out.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, lse


def bwd_workspace_size(q, k, heads_k_stride=1, grad_fp32=False) -> int:
    return int(library().ringattn_bwd_workspace_size(
        make_dims(q, k, 0, heads_k_stride, grad_fp32)))


def set_bwd_flush_interval(pairs: int) -> None:
    """(query tile, head) pairs after which the dK/dV kernel moves its
    tensor-memory sums to fp32 memory and restarts them; 0: never.
    Process-wide; size backward workspaces after changing it."""
    _check("ringattn_set_bwd_flush_interval", library().ringattn_set_bwd_flush_interval(int(pairs)))


def ringattn_bwd(q, k, v, out, lse, dout, cu_seqlens=None, num_shards=1,
                 shard_layout=CONTIGUOUS, causal=True, dq=None, dk=None, dv=None,
                 workspace=None, stream=None, heads_k_stride=1, grad_fp32=False,
                 kv_exchange=RING):
    """Ring-attention backward; returns (dq, dk, dv) (fp32 if grad_fp32)."""
    import torch
    _check_qkv(q, k, v)
    T, hq, d = q.shape
    _need(out, "out", q.shape, q.dtype)
    _need(dout, "dout", q.shape, q.dtype)
    _need(lse, "lse", (hq, T), torch.float32)
    gdt = torch.float32 if grad_fp32 else q.dtype
    dq = torch.empty(q.shape, dtype=gdt, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=gdt, device=k.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=gdt, device=v.device) if dv is None else dv
    _need(dq, "dq", q.shape, gdt)
    _need(dk, "dk", k.shape, gdt)
    _need(dv, "dv", v.shape, gdt)
    need = bwd_workspace_size(q, k, heads_k_stride, grad_fp32)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    cu_p, nseq, _keep = _cu_host(cu_seqlens)
    dims = make_dims(q, k, nseq, heads_k_stride, grad_fp32, kv_exchange)
    _check("ringattn_bwd", library().ringattn_bwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
        dout.data_ptr(), cu_p, dims, int(num_shards), int(shard_layout), int(bool(causal)),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return dq, dk, dv


def _rank_dims(q, k, total_tokens, num_seqs):
    """Whole-problem dims from one rank's local buffers ([T / P, H, D])."""
    _, hq, d = q.shape
    return ra_dims(int(total_tokens), num_seqs, hq, k.shape[1], d, _dtype_code(q), 1, 1, RING)


def fwd_rank_workspace_size(q, k, total_tokens, num_shards) -> int:
    return int(library().ringattn_fwd_rank_workspace_size(_rank_dims(q, k, total_tokens, 0),
                                                          int(num_shards)))


def bwd_rank_workspace_size(q, k, total_tokens, num_shards) -> int:
    return int(library().ringattn_bwd_rank_workspace_size(_rank_dims(q, k, total_tokens, 0),
                                                          int(num_shards)))


def ringattn_fwd_rank_step(q, k, v, cu_seqlens, total_tokens, num_shards, shard_layout, causal,
                           rank, step, o_acc, lse_acc, out, lse, workspace, stream=None):
    """One ring step of one rank on shard-local buffers (see ringattn.h)."""
    import torch
    _check_qkv(q, k, v)
    Tr, hq, d = q.shape
    ptr = lambda t: None if t is None else t.data_ptr()
    for t, n, shp, dt in ((o_acc, "o_acc", (Tr, hq, d), torch.float32),
                          (lse_acc, "lse_acc", (hq, Tr), torch.float32),
                          (out, "out", (Tr, hq, d), q.dtype), (lse, "lse", (hq, Tr), torch.float32)):
        if t is not None:
            _need(t, n, shp, dt)
    cu_p, nseq, _keep = _cu_host(cu_seqlens)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("ringattn_fwd_rank_step", library().ringattn_fwd_rank_step(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), cu_p, _rank_dims(q, k, total_tokens, nseq),
        int(num_shards), int(shard_layout), int(bool(causal)), int(rank), int(step), ptr(o_acc),
        ptr(lse_acc), ptr(out), ptr(lse), ptr(workspace), ws, _stream(stream)))


def ringattn_bwd_rank_step(q, k, v, out, lse, dout, cu_seqlens, total_tokens, num_shards,
                           shard_layout, causal, rank, step, dq, dk, dv, workspace, stream=None):
    """Backward of one ring step of one rank; fp32 dq, dk, dv (see ringattn.h)."""
    import torch
    _check_qkv(q, k, v)
    Tr, hq, d = q.shape
    _need(out, "out", q.shape, q.dtype)
    _need(dout, "dout", q.shape, q.dtype)
    _need(lse, "lse", (hq, Tr), torch.float32)
    _need(dq, "dq", q.shape, torch.float32)
    _need(dk, "dk", k.shape, torch.float32)
    _need(dv, "dv", v.shape, torch.float32)
    cu_p, nseq, _keep = _cu_host(cu_seqlens)
    _check("ringattn_bwd_rank_step", library().ringattn_bwd_rank_step(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
        dout.data_ptr(), cu_p, _rank_dims(q, k, total_tokens, nseq), int(num_shards),
        int(shard_layout), int(bool(causal)), int(rank), int(step), dq.data_ptr(),
        dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def attn_lse_merge(o_a, lse_a, o_b, lse_b, stream=None):
    """In-place log-sum-exp merge of (o_b, lse_b) into (o_a, lse_a)."""
    import torch
    _need(o_a, "o_a")
    _need(o_b, "o_b", o_a.shape, o_a.dtype)
    rows, heads, d = o_a.shape
    _need(lse_a, "lse_a", (heads, rows), torch.float32)
    _need(lse_b, "lse_b", (heads, rows), torch.float32)
    _check("attn_lse_merge", library().attn_lse_merge(
        o_a.data_ptr(), lse_a.data_ptr(), o_b.data_ptr(), lse_b.data_ptr(), rows, heads, d,
        _dtype_code(o_a), _stream(stream)))
    return o_a, lse_a


def ringattn_get_status(stream=None) -> int:
    """Synchronises the stream; returns and clears the kernel-side error word."""
    return int(library().ringattn_get_status(_stream(stream)))


def debug_report(stream=None):
    """(checks_compiled_in, site, index) of the first failed bounds check since
    the last call (site 0: none); only the debug build makes checks."""
    site, index = ctypes.c_longlong(0), ctypes.c_longlong(0)
    rc = library().ringattn_debug_report(_stream(stream), ctypes.byref(site), ctypes.byref(index))
    if rc < 0:
        raise RingAttnError("ringattn_debug_report", -4)
    return bool(rc), int(site.value), int(index.value)


def selftest_wait_timeout(stream=None) -> None:
    """Launches the failure-path self-test: one kernel wait that runs out
    after its time limit and records RA_ERR_TIMEOUT (read it with
    ringattn_get_status)."""
    _check("ringattn_selftest_wait_timeout",
           library().ringattn_selftest_wait_timeout(_stream(stream)))


def _plan(fn_name, item_fields, total_tokens, hq, hkv, num_shards, shard_layout, causal,
          cu_seqlens, heads_k_stride, kv_exchange=RING, extra=()):
    cu_p, nseq, _keep = _cu_host(cu_seqlens)
    dims = ra_dims(total_tokens, nseq, hq, hkv, 64, RA_FP32, heads_k_stride, 0, kv_exchange)
    ni, ns = ctypes.c_int(0), ctypes.c_int(0)
    fn = getattr(library(), fn_name)
    head = (cu_p, dims, num_shards, shard_layout, int(bool(causal))) + tuple(extra)
    code = fn(*head, None, 0, None, 0, ctypes.byref(ni), ctypes.byref(ns))
    if code not in (0, -6):
        raise RingAttnError(fn_name, code)
    items = np.zeros((max(ni.value, 1), item_fields), np.int32)
    segs = np.zeros((max(ns.value, 1), PLAN_SEG_FIELDS), np.int32)
    _check(fn_name, fn(*head, items.ctypes.data_as(_i32p), items.shape[0],
                       segs.ctypes.data_as(_i32p), segs.shape[0], ctypes.byref(ni),
                       ctypes.byref(ns)))
    return items[:ni.value], segs[:ns.value]


def plan_fwd(total_tokens, hq, hkv, num_shards, shard_layout, causal, cu_seqlens=None,
             heads_k_stride=1, kv_exchange=RING):
    """Host-only: the forward work list as (items [n,16], segments [m,4]) int32 arrays."""
    return _plan("ringattn_plan_fwd", PLAN_ITEM_FIELDS, total_tokens, hq, hkv, num_shards,
                 shard_layout, causal, cu_seqlens, heads_k_stride, kv_exchange)


def plan_fwd_fused(total_tokens, hq, hkv, num_shards, shard_layout, causal, num_sms,
                   cu_seqlens=None, heads_k_stride=1, kv_exchange=RING):
    """Host-only: the fused forward's work list on a GPU of num_sms SMs, in claim
    order, with long items split (items [n,16], segments [m,4])."""
    return _plan("ringattn_plan_fwd_fused", PLAN_ITEM_FIELDS, total_tokens, hq, hkv, num_shards,
                 shard_layout, causal, cu_seqlens, heads_k_stride, kv_exchange,
                 extra=(int(num_sms),))


def plan_bwd(total_tokens, hq, hkv, num_shards, shard_layout, causal, cu_seqlens=None,
             heads_k_stride=1, kv_exchange=RING):
    """Host-only: the key-side backward work list (items [n,8], segments [m,4])."""
    return _plan("ringattn_plan_bwd", PLAN_BWD_ITEM_FIELDS, total_tokens, hq, hkv, num_shards,
                 shard_layout, causal, cu_seqlens, heads_k_stride, kv_exchange)


def trace_enable(on: bool = True) -> None:
    """Start (or stop) recording every kernel launch of the library between
    two CUDA events on its launch stream."""
    _check("ringattn_trace_enable", library().ringattn_trace_enable(int(bool(on))))


def trace_collect() -> dict:
    """Waits for the recorded launches; returns {kernel: (launches, total_ms)}
    since the last collect and clears the record."""
    n = ctypes.c_int(0)
    buf = (ra_trace_entry * 64)()  # one entry per kernel name; the library has fewer
    _check("ringattn_trace_collect", library().ringattn_trace_collect(buf, 64, ctypes.byref(n)))
    return {buf[i].kernel.decode(): (int(buf[i].launches), float(buf[i].total_ms))
            for i in range(n.value)}


def _ssd_dims(x, B):
    T, H, P = x.shape
    return ssd_dims(T, H, P, B.shape[2], B.shape[1])


def ssd_cp_workspace_size(x, B, num_shards) -> int:
    return int(library().ssd_cp_workspace_size(_ssd_dims(x, B), int(num_shards)))


def ssd_cp_fwd(x, dt, A, B, C, D=None, position_ids=None, num_shards=1, y=None,
               final_state=None, workspace=None, stream=None, want_final_state=False):
    """Context-parallel Mamba2 selective scan (fp32): returns (y [T,H,64],
    final state [H,64,N] or None).  position_ids: int32 device tensor [T] or
    None; a token at position 0 starts a packed sample."""
    import torch
    for t, n in ((x, "x"), (dt, "dt"), (A, "A"), (B, "B"), (C, "C")):
        _need(t, n, dtype=torch.float32)
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    _need(dt, "dt", (T, H))
    _need(A, "A", (H,))
    _need(C, "C", B.shape)
    if D is not None:
        _need(D, "D", (H,), torch.float32)
    if position_ids is not None:
        _need(position_ids, "position_ids", (T,), torch.int32)
    if y is None:
        y = torch.empty_like(x)
    _need(y, "y", x.shape, torch.float32)
    if final_state is None and want_final_state:
        final_state = torch.empty(H, P, N, dtype=torch.float32, device=x.device)
    if final_state is not None:
        _need(final_state, "final_state", (H, P, N), torch.float32)
    need = ssd_cp_workspace_size(x, B, num_shards)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    ptr = lambda t: None if t is None else t.data_ptr()
    _check("ssd_cp_fwd", library().ssd_cp_fwd(
        x.data_ptr(), dt.data_ptr(), A.data_ptr(), B.data_ptr(), C.data_ptr(), ptr(D),
        ptr(position_ids), _ssd_dims(x, B), int(num_shards), y.data_ptr(), ptr(final_state),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream)))
    return y, final_state
