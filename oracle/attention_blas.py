"""Exact softmax attention in fp64 with library matrix products.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may use this module; nothing on the product path
imports it, and it imports nothing from the product package.

It computes the same definition as ``attention_fp64.c`` -- attention over the
WHOLE, unsharded sequence, which ring attention reaches by re-ordering the sum
(axolotl "Sequence Parallelism" page, introduction and "Implementation
Details"; aicassindra "tm_sp_math", "Context parallelism is the axis that is
independent": every query must see every key) -- but each sum over d, over
keys or over queries is one fp64 matrix product of the CPU math library
(``torch.matmul`` on float64 tensors).  That makes a whole head of 32K tokens
a matter of seconds, so the GPU parity tests can compare every row of the
full-size workloads instead of a sample.  For query row i of head h
(key/value head g = h // (Hq / Hkv)):

  visible set  V(i) = { j : doc(j) = doc(i), and j <= i when causal }, doc()
               from cu_seqlens (positions restart per packed sample: axolotl
               page, "Sample Packing with Sequence Parallelism"); no
               cu_seqlens = one document.  key_allowed (forward only)
               removes keys from every V(i): one ring step's partial result.
  scores       S_ij = scale q_i . k_j                     (matrix product)
  lse          m_i = max_{j in V(i)} S_ij,  lse_i = m_i + ln sum_{j in V(i)} e^(S_ij - m_i)
  output       O_i = sum_{j in V(i)} e^(S_ij - lse_i) v_j   (matrix product)
  backward     P_ij = e^(S_ij - lse_i),  dP_ij = dO_i . v_j,
               D_i = sum_j P_ij dP_ij  (from the definition, not via O),
               dS_ij = P_ij (dP_ij - D_i),
               dQ_i = scale sum_j dS_ij k_j,
               dK_j = scale sum_{h in group g} sum_i dS_ij q_i,
               dV_j = sum_{h in group g} sum_i P_ij dO_i.

The query-side quantities (lse, D, dQ) are computed first, row by row (a
block of rows per matrix product), and the key-side sums (dK, dV) afterwards,
key by key, from those row statistics -- the same two passes as the C oracle.
Scores are formed only for keys of the documents a block of rows can reach
(and, when causal, only up to the block's last row); every other key is
invisible by definition, so leaving it out changes no result.  Inside that
span the visible set is applied as an explicit mask built from doc() and the
causal rule.  Rows with no visible key get O = 0 and lse = -inf.  Heads that
a call is not asked for are NaN in its outputs, so they cannot be mistaken
for results.
"""
from __future__ import annotations

import math

import numpy as np
import torch

# scores held at once: rows per block x keys in the block's span
_BLOCK_ELEMS = 1 << 24


def _f64(x) -> torch.Tensor:
    """CPU float64 tensor of an array or tensor (fp32 or bf16 values widened)."""
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu").to(torch.float64)
    return torch.from_numpy(np.asarray(x, dtype=np.float64))


def _docs(T: int, cu_seqlens):
    """doc(t) for every token, and each document's [start, end)."""
    if cu_seqlens is None:
        cu = np.array([0, T], np.int64)
    else:
        cu = np.asarray([int(c) for c in cu_seqlens], np.int64)
        if cu.ndim != 1 or cu.size < 2 or cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
            raise ValueError("cu_seqlens must run from 0 to T without decreasing")
    # the document whose range [cu[d], cu[d+1]) holds t
    doc = np.searchsorted(cu, np.arange(T), side="right") - 1
    start = cu[doc]
    end = cu[doc + 1]
    return torch.from_numpy(doc), start, end


def _row_blocks(T: int, span: int):
    step = max(16, min(1024, _BLOCK_ELEMS // max(1, span)))
    for r0 in range(0, T, step):
        yield r0, min(T, r0 + step)


def _mask(doc, rows: slice, keys: slice, causal: bool, key_allowed=None) -> torch.Tensor:
    """V(i) restricted to the given rows and keys, as a boolean matrix."""
    vis = doc[rows][:, None] == doc[keys][None, :]
    if causal:
        i = torch.arange(rows.start, rows.stop)[:, None]
        j = torch.arange(keys.start, keys.stop)[None, :]
        vis &= j <= i
    if key_allowed is not None:
        vis &= key_allowed[keys][None, :]
    return vis


def _row_stats(S: torch.Tensor, vis: torch.Tensor):
    """lse of each row of scores over its visible set (max first, then the
    shifted sum), and the weights P_ij = e^(S_ij - m_i) / sum_j e^(S_ij - m_i)
    = e^(S_ij - lse_i), 0 outside the visible set.  S is overwritten."""
    S.masked_fill_(~vis, -math.inf)
    m = S.max(dim=1).values
    empty = ~torch.isfinite(m)
    m = torch.where(empty, torch.zeros_like(m), m)
    E = S.sub_(m[:, None]).exp_()          # e^(S - m); hidden keys give e^-inf = 0
    z = E.sum(dim=1)
    lse = torch.where(empty, torch.full_like(m, -math.inf), m + torch.log(z))
    P = E.div_(torch.where(empty, torch.ones_like(z), z)[:, None])
    return lse, P


def _check_shapes(q, k, v):
    T, hq, d = q.shape
    if k.shape[0] != T or k.shape[2] != d or v.shape != k.shape or hq % k.shape[1]:
        raise ValueError("shapes: q [T,Hq,D], k/v [T,Hkv,D], Hq % Hkv == 0")
    return T, hq, k.shape[1], d


def _spans(start, end, causal, r0, r1):
    """Keys any row of [r0, r1) may see: the documents of its rows."""
    k0 = int(start[r0])
    k1 = r1 if causal else int(end[r1 - 1])
    return k0, k1


def attention_fwd(q, k, v, *, causal, cu_seqlens=None, scale=None, heads=None,
                  key_allowed=None):
    """O [T, Hq, D] and lse [Hq, T] (natural log), fp64 numpy arrays.

    heads: the query heads to compute (default all); the others are NaN.
    key_allowed: optional boolean array of T entries removing keys from every
    visible set (one ring step's partial result when it marks that step's
    K/V chunks)."""
    T, hq, hkv, d = _check_shapes(q, k, v)
    G = hq // hkv
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    doc, start, end = _docs(T, cu_seqlens)
    ka = None
    if key_allowed is not None:
        ka = torch.from_numpy(np.asarray(key_allowed, dtype=bool).copy())
        if ka.numel() != T:
            raise ValueError("key_allowed must have T entries")
    hl = list(range(hq)) if heads is None else [int(h) for h in heads]
    o = np.full((T, hq, d), np.nan)
    lse = np.full((hq, T), np.nan)
    if T == 0:
        return o, lse
    for h in hl:
        g = h // G
        Qh = _f64(q[:, h, :]).contiguous()
        KgT = _f64(k[:, g, :]).T.contiguous()   # [D, T]
        Vg = _f64(v[:, g, :]).contiguous()
        for r0, r1 in _row_blocks(T, T):
            k0, k1 = _spans(start, end, causal, r0, r1)
            rows, keys = slice(r0, r1), slice(k0, k1)
            S = (Qh[rows] @ KgT[:, keys]).mul_(sc)
            vis = _mask(doc, rows, keys, causal, ka)
            L, P = _row_stats(S, vis)
            o[r0:r1, h, :] = (P @ Vg[keys]).numpy()
            lse[h, r0:r1] = L.numpy()
    return o, lse


def attention_bwd(q, k, v, dout, *, causal, cu_seqlens=None, scale=None, kv_heads=None,
                  return_out=False):
    """dQ [T, Hq, D], dK [T, Hkv, D], dV [T, Hkv, D], D [Hq, T], lse [Hq, T]
    (and O [T, Hq, D] last when return_out is set: the forward output of the
    same rows, O_i = sum_j P_ij v_j).

    kv_heads: the key/value heads to compute (default all) -- dK, dV of those
    heads and dQ, D, lse (and O) of every query head of their groups; the
    rest NaN."""
    T, hq, hkv, d = _check_shapes(q, k, v)
    if tuple(dout.shape) != (T, hq, d):
        raise ValueError("dout must match q")
    G = hq // hkv
    sc = 1.0 / math.sqrt(d) if scale is None else float(scale)
    doc, start, end = _docs(T, cu_seqlens)
    gl = list(range(hkv)) if kv_heads is None else [int(g) for g in kv_heads]
    dq = np.full((T, hq, d), np.nan)
    dk = np.full((T, hkv, d), np.nan)
    dv = np.full((T, hkv, d), np.nan)
    Dvec = np.full((hq, T), np.nan)
    lse = np.full((hq, T), np.nan)
    o = np.full((T, hq, d), np.nan) if return_out else None
    if T == 0:
        return (dq, dk, dv, Dvec, lse, o) if return_out else (dq, dk, dv, Dvec, lse)
    for g in gl:
        Kg = _f64(k[:, g, :]).contiguous()
        KgT = Kg.T.contiguous()                  # [D, T]
        VgT = _f64(v[:, g, :]).T.contiguous()    # [D, T]
        Qs, dOs, Ls, Ds = {}, {}, {}, {}
        # query side: lse_i, D_i and dQ_i, row by row
        for h in range(g * G, (g + 1) * G):
            Qh = _f64(q[:, h, :]).contiguous()
            dOh = _f64(dout[:, h, :]).contiguous()
            Lh = torch.empty(T, dtype=torch.float64)
            Dh = torch.empty(T, dtype=torch.float64)
            for r0, r1 in _row_blocks(T, T):
                k0, k1 = _spans(start, end, causal, r0, r1)
                rows, keys = slice(r0, r1), slice(k0, k1)
                S = (Qh[rows] @ KgT[:, keys]).mul_(sc)
                vis = _mask(doc, rows, keys, causal)
                L, P = _row_stats(S, vis)
                if return_out:
                    o[r0:r1, h, :] = (P @ VgT[:, keys].T).numpy()
                dP = dOh[rows] @ VgT[:, keys]
                Dr = (P * dP).sum(dim=1)
                dS = dP.sub_(Dr[:, None]).mul_(P)      # P (dP - D)
                dq[r0:r1, h, :] = (dS @ Kg[keys]).mul_(sc).numpy()
                Lh[r0:r1] = L
                Dh[r0:r1] = Dr
            Qs[h], dOs[h], Ls[h], Ds[h] = Qh, dOh, Lh, Dh
            lse[h] = Lh.numpy()
            Dvec[h] = Dh.numpy()
        # key side: dK_j, dV_j summed over the group's heads, key by key
        for j0, j1 in _row_blocks(T, T):
            # queries that may see a key of [j0, j1): its documents' rows
            # (and, when causal, only rows from j0 on)
            i0 = j0 if causal else int(start[j0])
            i1 = int(end[j1 - 1])
            rows, keys = slice(i0, i1), slice(j0, j1)
            hidden = ~_mask(doc, rows, keys, causal)
            acc_k = torch.zeros(j1 - j0, d, dtype=torch.float64)
            acc_v = torch.zeros(j1 - j0, d, dtype=torch.float64)
            for h in range(g * G, (g + 1) * G):
                S = (Qs[h][rows] @ KgT[:, keys]).mul_(sc)
                L = Ls[h][rows]
                L = torch.where(torch.isfinite(L), L, torch.zeros_like(L))
                # P = e^(S - lse); hidden pairs give e^-inf = 0
                P = S.masked_fill_(hidden, -math.inf).sub_(L[:, None]).exp_()
                dP = dOs[h][rows] @ VgT[:, keys]
                dS = dP.sub_(Ds[h][rows][:, None]).mul_(P)   # P (dP - D)
                acc_k += dS.T @ Qs[h][rows]
                acc_v += P.T @ dOs[h][rows]
            dk[j0:j1, g, :] = acc_k.mul_(sc).numpy()
            dv[j0:j1, g, :] = acc_v.numpy()
    return (dq, dk, dv, Dvec, lse, o) if return_out else (dq, dk, dv, Dvec, lse)
