"""fp64 CPU oracle of exact softmax attention (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the bench's ``cpu_baseline``
leg may import this package.  The product path (the CUDA library and its
binding) never imports, links or calls it, and it imports nothing from the
product package.

The arithmetic lives in ``attention_fp64.c`` and ``ssd_fp64.c`` (plain C,
OpenMP over rows / heads); this module compiles them with gcc on first use and
marshals numpy/torch arrays to them.  ``oracle.blas`` (``attention_blas.py``)
computes the same attention definition with fp64 library matrix products, fast
enough to check every row of the full-size workloads; it is pinned by the same
checks as the C oracle.
Every function computes the plain definition of attention over the whole,
unsharded sequence (the ring schedule is an exact re-ordering of that sum,
axolotl "Sequence Parallelism" page, introduction and "Implementation
Details"), plus the log-sum-exp merge that aggregates ring steps.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "attention_fp64.c"), os.path.join(_HERE, "ssd_fp64.c")]
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)
_up = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc -O2 -fopenmp (no fast-math: IEEE fp64)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(f) for f in _SRCS))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                        "-std=c11", "-o", tmp] + _SRCS + ["-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_fwd_rows.argtypes = [
                _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, _ip, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                _up, ctypes.c_int, _ip, _ip, _dp, _dp]
            lib.oracle_bwd_rows.argtypes = [
                _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, _ip, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                ctypes.c_int, _ip, _ip, _dp, _dp, _dp]
            lib.oracle_bwd_keys.argtypes = [
                _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, _ip, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                ctypes.c_int, _ip, _ip, _dp, _dp]
            lib.oracle_lse_merge.argtypes = [ctypes.c_int, ctypes.c_int,
                                             _dp, _dp, _dp, _dp]
            lib.oracle_lse_merge.restype = None
            lib.oracle_ssd_scan.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _ip, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, _dp, _dp, _dp]
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle uses (all host cores unless OMP_NUM_THREADS)."""
    return int(_load().oracle_num_threads())


def _f64(x) -> np.ndarray:
    """Widen a torch tensor or array (fp32 or bf16 values) to C-contiguous fp64."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        x = x.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a: np.ndarray, typ):
    return a.ctypes.data_as(typ)


def _cu(cu_seqlens, T):
    if cu_seqlens is None:
        return None, 0
    cu = _i32(cu_seqlens)
    if cu.ndim != 1 or cu.size < 2 or cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must run from 0 to T without decreasing")
    return cu, cu.size - 1


def _shapes(q, k, v):
    T, hq, d = q.shape
    Tk, hkv, dk = k.shape
    if Tk != T or dk != d or v.shape != k.shape or hq % hkv:
        raise ValueError("shapes: q [T,Hq,D], k/v [T,Hkv,D], Hq % Hkv == 0")
    return T, hq, hkv, d


def _check(rc):
    if rc != 0:
        raise RuntimeError(f"oracle returned {rc}")


def fwd_rows(q, k, v, heads, rows, *, causal, cu_seqlens=None, scale=None,
             key_allowed=None):
    """O (n, D) and lse (n,) for the n (head, row) pairs given.

    key_allowed (bool array of length T) restricts the keys further: that is
    one ring step's partial result when it marks one step's KV chunks.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, hq, hkv, d = _shapes(q, k, v)
    cu, nseq = _cu(cu_seqlens, T)
    hs, is_ = _i32(heads).ravel(), _i32(rows).ravel()
    n = hs.size
    if is_.size != n or (n and (hs.min() < 0 or hs.max() >= hq or is_.min() < 0 or is_.max() >= T)):
        raise ValueError("bad (head, row) list")
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    ka = None
    if key_allowed is not None:
        ka = np.ascontiguousarray(np.asarray(key_allowed, dtype=np.uint8))
        if ka.size != T:
            raise ValueError("key_allowed must have T entries")
    o = np.zeros((n, d), np.float64)
    lse = np.zeros(n, np.float64)
    _check(_load().oracle_fwd_rows(
        _ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), T, hq, hkv, d,
        None if cu is None else _ptr(cu, _ip), nseq, int(bool(causal)), sc,
        None if ka is None else _ptr(ka, _up), n, _ptr(hs, _ip), _ptr(is_, _ip),
        _ptr(o, _dp), _ptr(lse, _dp)))
    return o, lse


def attention_fwd(q, k, v, *, causal, cu_seqlens=None, scale=None,
                  key_allowed=None, heads=None):
    """Full forward: O [T, Hq, D] and lse [Hq, T] (natural log), fp64.

    heads: optional list of q heads to compute; the others stay zero (O) and
    NaN (lse), so a caller cannot mistake them for results.
    """
    T, hq, d = q.shape
    hl = list(range(hq)) if heads is None else [int(h) for h in heads]
    hs = np.repeat(np.asarray(hl, np.int32), T)
    is_ = np.tile(np.arange(T, dtype=np.int32), len(hl))
    o_r, l_r = fwd_rows(q, k, v, hs, is_, causal=causal, cu_seqlens=cu_seqlens,
                        scale=scale, key_allowed=key_allowed)
    o = np.zeros((T, hq, d), np.float64)
    lse = np.full((hq, T), np.nan, np.float64)
    for n, h in enumerate(hl):
        o[:, h, :] = o_r[n * T:(n + 1) * T]
        lse[h, :] = l_r[n * T:(n + 1) * T]
    return o, lse


def bwd_rows(q, k, v, dout, heads, rows, *, causal, cu_seqlens=None, scale=None):
    """dQ (n, D), D_i (n,) and lse (n,) for the n (head, row) pairs given."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
    T, hq, hkv, d = _shapes(q, k, v)
    if do.shape != q.shape:
        raise ValueError("dout must match q")
    cu, nseq = _cu(cu_seqlens, T)
    hs, is_ = _i32(heads).ravel(), _i32(rows).ravel()
    n = hs.size
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = np.zeros((n, d), np.float64)
    Dv = np.zeros(n, np.float64)
    lse = np.zeros(n, np.float64)
    _check(_load().oracle_bwd_rows(
        _ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(do, _dp), T, hq, hkv, d,
        None if cu is None else _ptr(cu, _ip), nseq, int(bool(causal)), sc, n,
        _ptr(hs, _ip), _ptr(is_, _ip), _ptr(dq, _dp), _ptr(Dv, _dp), _ptr(lse, _dp)))
    return dq, Dv, lse


def bwd_keys(q, k, v, dout, kv_heads, keys, *, causal, cu_seqlens=None, scale=None):
    """dK (n, D) and dV (n, D), summed over each kv head's q-head group."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
    T, hq, hkv, d = _shapes(q, k, v)
    cu, nseq = _cu(cu_seqlens, T)
    gs, js = _i32(kv_heads).ravel(), _i32(keys).ravel()
    n = gs.size
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dk = np.zeros((n, d), np.float64)
    dv = np.zeros((n, d), np.float64)
    _check(_load().oracle_bwd_keys(
        _ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(do, _dp), T, hq, hkv, d,
        None if cu is None else _ptr(cu, _ip), nseq, int(bool(causal)), sc, n,
        _ptr(gs, _ip), _ptr(js, _ip), _ptr(dk, _dp), _ptr(dv, _dp)))
    return dk, dv


def attention_bwd(q, k, v, dout, *, causal, cu_seqlens=None, scale=None):
    """Full backward: dQ [T,Hq,D], dK [T,Hkv,D], dV [T,Hkv,D], D [Hq,T], lse [Hq,T]."""
    T, hq, d = q.shape
    hkv = k.shape[1]
    hs = np.repeat(np.arange(hq, dtype=np.int32), T)
    is_ = np.tile(np.arange(T, dtype=np.int32), hq)
    dq_r, D_r, l_r = bwd_rows(q, k, v, dout, hs, is_, causal=causal,
                              cu_seqlens=cu_seqlens, scale=scale)
    gs = np.repeat(np.arange(hkv, dtype=np.int32), T)
    js = np.tile(np.arange(T, dtype=np.int32), hkv)
    dk_r, dv_r = bwd_keys(q, k, v, dout, gs, js, causal=causal,
                          cu_seqlens=cu_seqlens, scale=scale)
    dq = dq_r.reshape(hq, T, d).transpose(1, 0, 2).copy()
    dk = dk_r.reshape(hkv, T, d).transpose(1, 0, 2).copy()
    dv = dv_r.reshape(hkv, T, d).transpose(1, 0, 2).copy()
    return dq, dk, dv, D_r.reshape(hq, T), l_r.reshape(hq, T)


def lse_merge(o_a, lse_a, o_b, lse_b):
    """Merged (O, lse) of two partial results over disjoint key sets.

    o_x: [..., D] rows; lse_x: matching [...] rows.  Returns new arrays.
    """
    oa = _f64(o_a).copy()
    la = _f64(lse_a).copy()
    ob, lb = _f64(o_b), _f64(lse_b)
    d = oa.shape[-1]
    n = la.size
    if oa.size != n * d or ob.size != n * d or lb.size != n:
        raise ValueError("merge operands disagree in shape")
    oa2, la2 = oa.reshape(n, d), la.reshape(n)
    ob2 = np.ascontiguousarray(ob.reshape(n, d))
    lb2 = np.ascontiguousarray(lb.reshape(n))
    _load().oracle_lse_merge(n, d, _ptr(oa2, _dp), _ptr(la2, _dp),
                             _ptr(ob2, _dp), _ptr(lb2, _dp))
    return oa2.reshape(oa.shape), la2.reshape(la.shape)


def ssd_scan(x, dt, A, B, C, D=None, position_ids=None, h0=None):
    """Mamba2 selective scan over the whole sequence, fp64 (ssd_fp64.c).

    x [T, H, P], dt [T, H], A [H], B and C [T, G, N], D [H] or None,
    position_ids [T] or None (a token with position 0 starts a packed sample
    and resets the state), h0 [H, P, N] or None.  Returns (y [T, H, P],
    final state [H, P, N]).
    """
    x, dt, A, B, C = _f64(x), _f64(dt), _f64(A), _f64(B), _f64(C)
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    if dt.shape != (T, H) or A.shape != (H,) or B.shape != (T, G, N) or C.shape != B.shape \
            or H % G:
        raise ValueError("ssd_scan shapes: x [T,H,P], dt [T,H], A [H], B, C [T,G,N]")
    Dd = None if D is None else _f64(D)
    pos = None if position_ids is None else _i32(position_ids)
    h0d = None if h0 is None else _f64(h0)
    y = np.zeros((T, H, P), np.float64)
    hT = np.zeros((H, P, N), np.float64)
    _check(_load().oracle_ssd_scan(
        _ptr(x, _dp), _ptr(dt, _dp), _ptr(A, _dp), _ptr(B, _dp), _ptr(C, _dp),
        None if Dd is None else _ptr(Dd, _dp), None if pos is None else _ptr(pos, _ip),
        T, H, P, N, G, None if h0d is None else _ptr(h0d, _dp), _ptr(y, _dp), _ptr(hT, _dp)))
    return y, hT


from . import attention_blas as blas  # noqa: E402  (fp64 matrix-product oracle)
