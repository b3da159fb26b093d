"""Multi-GPU ring attention: the host side of the ring.

The pages deploy ring attention with one rank per GPU: each rank keeps its
own query rows (and, in the backward, its rows of O, dO and lse), while the
K/V shards travel around the ring so that no device ever holds the whole
sequence (aicassindra "tm_sp_math", "Context parallelism is the axis that is
independent"; axolotl "Sequence Parallelism" page, introduction and
"Implementation Details": results aggregated through a ring communication
pattern).  At ring step s rank r holds the K/V shard of rank (r - s) mod P.
While the step computes, the rank passes that shard on to rank (r + 1) mod P
and receives the next one from rank (r - 1) mod P into a second buffer
(double buffering), so the transfer of step s + 1's shard overlaps step s's
compute.  The backward also carries the shard's dK/dV accumulators along the
ring and, after the last step, returns them to the shard's owner.

This module only moves buffers and orders the steps: every step's attention
runs in the library's kernels (ringattn_fwd_rank_step and
ringattn_bwd_rank_step, which fold each step into the rank's running result
with the log-sum-exp merge).  Two transports share the schedule:

* ring_fwd / ring_bwd: one process per rank, torch.distributed point-to-point
  operations on the default process group (NCCL between GPUs; the
  bookkeeping works with any backend);
* EmulatedRing (and emulate_ring_fwd / emulate_ring_bwd on top of it): all P
  ranks in one process on one GPU, each rank with its own device buffers and
  its own stream, the shards passed by device-to-device copies ordered with
  events -- the same schedule, to check and time it without P GPUs.

Buffers of rank r hold its rows back to back: CONTIGUOUS tokens
[r T/P, (r+1) T/P); ZIGZAG chunk r then chunk 2P-1-r of 2P equal chunks.
"""
from __future__ import annotations

from . import CONTIGUOUS, ZIGZAG, ringattn_bwd_rank_step, ringattn_fwd_rank_step
from . import bwd_rank_workspace_size, fwd_rank_workspace_size


def rank_rows(total_tokens: int, num_shards: int, layout: int, rank: int):
    """Global token ranges [a, b) of rank `rank`'s buffer rows, in buffer order."""
    T, P = int(total_tokens), int(num_shards)
    if layout == CONTIGUOUS:
        if T % P:
            raise ValueError("total_tokens must divide by num_shards")
        C = T // P
        return [(rank * C, (rank + 1) * C)]
    if layout != ZIGZAG or T % (2 * P):
        raise ValueError("ZIGZAG needs total_tokens divisible by 2 * num_shards")
    C = T // (2 * P)
    return [(rank * C, (rank + 1) * C), ((2 * P - 1 - rank) * C, (2 * P - rank) * C)]


def shard(x, num_shards: int, layout: int, rank: int):
    """Rank `rank`'s rows (dim 0) of a whole-sequence tensor, as a new tensor."""
    import torch
    return torch.cat([x[a:b] for a, b in rank_rows(x.shape[0], num_shards, layout, rank)]).contiguous()


def unshard(parts, num_shards: int, layout: int, dim: int = 0):
    """The whole-sequence tensor from every rank's rows (inverse of shard);
    dim is the token dimension (1 for lse [H, T])."""
    import torch
    Tr = parts[0].shape[dim]
    T = Tr * num_shards
    shape = list(parts[0].shape)
    shape[dim] = T
    out = torch.empty(shape, dtype=parts[0].dtype, device=parts[0].device)
    for r, part in enumerate(parts):
        off = 0
        for a, b in rank_rows(T, num_shards, layout, r):
            out.narrow(dim, a, b - a).copy_(part.narrow(dim, off, b - a))
            off += b - a
    return out


# ------------------------------------------------------------ one rank's state

class FwdRank:
    """One rank's forward on its GPU: the running (O, lse) and the step
    workspace; called once per ring step with the K/V shard it holds."""

    def __init__(self, q, total_tokens, num_shards, layout, causal, rank, cu_seqlens=None):
        import torch
        self.q, self.T, self.P, self.layout, self.causal = q, total_tokens, num_shards, layout, causal
        self.rank, self.cu = rank, cu_seqlens
        Tr, hq, d = q.shape
        f32 = dict(dtype=torch.float32, device=q.device)
        self.o_acc = torch.empty(Tr, hq, d, **f32)
        self.lse_acc = torch.empty(hq, Tr, **f32)
        self.out = torch.empty_like(q)
        self.lse = torch.empty(hq, Tr, **f32)
        self.ws = None

    def __call__(self, step, k, v, stream=None):
        import torch
        if self.ws is None:
            n = fwd_rank_workspace_size(self.q, k, self.T, self.P)
            self.ws = torch.empty(max(n, 16), dtype=torch.uint8, device=self.q.device)
        ringattn_fwd_rank_step(self.q, k, v, self.cu, self.T, self.P, self.layout, self.causal,
                               self.rank, step, self.o_acc, self.lse_acc, self.out, self.lse,
                               self.ws, stream)

    def result(self):
        return self.out, self.lse


class BwdRank:
    """One rank's backward on its GPU: dq of its rows (fp32) and the D_i
    workspace; called once per ring step with the K/V shard it holds and that
    shard's dK/dV accumulators."""

    def __init__(self, q, out, lse, dout, total_tokens, num_shards, layout, causal, rank,
                 cu_seqlens=None):
        import torch
        self.q, self.out, self.lse, self.dout = q, out, lse, dout
        self.T, self.P, self.layout, self.causal = total_tokens, num_shards, layout, causal
        self.rank, self.cu = rank, cu_seqlens
        self.dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        self.ws = None

    def __call__(self, step, k, v, dk, dv, stream=None):
        import torch
        if self.ws is None:
            n = bwd_rank_workspace_size(self.q, k, self.T, self.P)
            self.ws = torch.empty(max(n, 16), dtype=torch.uint8, device=self.q.device)
        ringattn_bwd_rank_step(self.q, k, v, self.out, self.lse, self.dout, self.cu, self.T,
                               self.P, self.layout, self.causal, self.rank, step, self.dq, dk, dv,
                               self.ws, stream)


# ------------------------------------------------- one process per rank

def _pass_on(send, recv, rank, world):
    """Posts the sends of `send` to the next rank and the receives into
    `recv` from the previous rank; returns the requests to wait on."""
    import torch.distributed as dist
    nxt, prv = (rank + 1) % world, (rank - 1) % world
    ops = [dist.P2POp(dist.isend, t, nxt) for t in send]
    ops += [dist.P2POp(dist.irecv, t, prv) for t in recv]
    return dist.batch_isend_irecv(ops)


def ring_fwd(q, k, v, *, total_tokens, layout, causal, cu_seqlens=None, rank_step=None):
    """Ring forward of this process's rank over the default process group.

    q, k, v: this rank's rows ([T/P, H, D]).  Returns this rank's
    (out [T/P, Hq, D], lse [Hq, T/P]).  rank_step: the per-step computation
    (default FwdRank, the library's kernels); anything with the same call and
    result() works, which is how the schedule is tested without a GPU."""
    import torch
    import torch.distributed as dist
    P, r = dist.get_world_size(), dist.get_rank()
    if rank_step is None:
        rank_step = FwdRank(q, total_tokens, P, layout, causal, r, cu_seqlens)
    bufs = [(torch.empty_like(k), torch.empty_like(v)) for _ in range(2 if P > 1 else 0)]
    cur_k, cur_v = k, v
    for s in range(P):
        reqs = []
        if s + 1 < P:   # the next shard travels while this step computes
            reqs = _pass_on([cur_k, cur_v], list(bufs[s % 2]), r, P)
        rank_step(s, cur_k, cur_v)
        for req in reqs:
            req.wait()
        if s + 1 < P:
            cur_k, cur_v = bufs[s % 2]
    return rank_step.result()


def ring_bwd(q, k, v, out, lse, dout, *, total_tokens, layout, causal, cu_seqlens=None,
             rank_step=None):
    """Ring backward of this process's rank.  Returns fp32 (dq of this rank's
    rows, dk and dv of this rank's keys).  K/V travel as in the forward; each
    shard's dK/dV accumulators follow it once its step has added to them, and
    the finished ones go back to their owner after the last step."""
    import torch
    import torch.distributed as dist
    P, r = dist.get_world_size(), dist.get_rank()
    if rank_step is None:
        rank_step = BwdRank(q, out, lse, dout, total_tokens, P, layout, causal, r, cu_seqlens)
    f32 = dict(dtype=torch.float32, device=k.device)
    cur = [k, v, torch.empty(k.shape, **f32), torch.empty(v.shape, **f32)]
    bufs = [[torch.empty_like(k), torch.empty_like(v), torch.empty(k.shape, **f32),
             torch.empty(v.shape, **f32)] for _ in range(2 if P > 1 else 0)]
    for s in range(P):
        reqs = []
        if s + 1 < P:   # K/V of the next step travel during this step
            reqs = _pass_on(cur[:2], bufs[s % 2][:2], r, P)
        rank_step(s, *cur)
        if s + 1 < P:   # then the accumulators this step has added to
            reqs += _pass_on(cur[2:], bufs[s % 2][2:], r, P)
        for req in reqs:
            req.wait()
        if s + 1 < P:
            cur = bufs[s % 2]
    if P == 1:
        return rank_step.dq, cur[2], cur[3]
    # after step P-1 this rank holds the finished dK/dV of rank r + 1
    dk, dv = torch.empty(k.shape, **f32), torch.empty(v.shape, **f32)
    for req in _pass_on(cur[2:], [dk, dv], r, P):
        req.wait()
    return rank_step.dq, dk, dv


# --------------------------------------- every rank on one GPU (emulation)

class EmulatedRing:
    """The multi-GPU ring with all P ranks on this GPU, set up once and run as
    often as wanted.  Each rank holds its own rows (copied in here), its own
    receive buffers (two per field: double buffering) and its own stream; the
    shards move by device-to-device copies on the sender's stream, ordered by
    events -- the schedule of ring_fwd / ring_bwd without P GPUs.

    fwd() returns every rank's (out, lse) rows; bwd(), after
    prepare_bwd(out, lse, dout), every rank's fp32 (dq, dk, dv) rows."""

    def __init__(self, q, k, v, *, num_shards, layout, causal, cu_seqlens=None):
        import torch
        P, T = num_shards, q.shape[0]
        self.P, self.T, self.layout, self.causal, self.cu = P, T, layout, causal, cu_seqlens
        self.kv = [[shard(k, P, layout, r), shard(v, P, layout, r)] for r in range(P)]
        self.fwd_ranks = [FwdRank(shard(q, P, layout, r), T, P, layout, causal, r, cu_seqlens)
                          for r in range(P)]
        self.fwd_bufs = [[[torch.empty_like(t) for t in self.kv[r]] for _ in range(2)]
                         for r in range(P)]
        self.streams = [torch.cuda.Stream(device=q.device) for _ in range(P)]
        self.bwd_ranks = None

    def _run(self, ranks, cur, bufs, fields):
        """The P ring steps: every rank computes step s on its stream, then
        passes what it holds on to the next rank (none after the last step)."""
        import torch
        P = self.P
        start = torch.cuda.current_stream(self.streams[0].device)
        for st in self.streams:
            st.wait_stream(start)
        for s in range(P):
            computed = [torch.cuda.Event() for _ in range(P)]
            for r in range(P):
                with torch.cuda.stream(self.streams[r]):
                    ranks[r](s, *cur[r], stream=self.streams[r])
                    computed[r].record(self.streams[r])
            if s + 1 < P:
                _emulated_pass_on(cur, bufs, s, self.streams, computed, fields)
        for st in self.streams:
            start.wait_stream(st)

    def fwd(self):
        self._run(self.fwd_ranks, [list(kv) for kv in self.kv], self.fwd_bufs, range(2))
        return [rk.result() for rk in self.fwd_ranks]

    def prepare_bwd(self, out, lse, dout):
        """The backward's per-rank rows of the whole-sequence forward results
        out [T, Hq, D], lse [Hq, T] and of dout, and its buffers."""
        import torch
        P, layout = self.P, self.layout
        self.bwd_ranks = [BwdRank(self.fwd_ranks[r].q, shard(out, P, layout, r),
                                  shard(lse.t(), P, layout, r).t().contiguous(),
                                  shard(dout, P, layout, r), self.T, P, layout, self.causal, r,
                                  self.cu) for r in range(P)]
        f32 = dict(dtype=torch.float32, device=out.device)
        self.dkv = [[torch.empty(kv[0].shape, **f32), torch.empty(kv[1].shape, **f32)]
                    for kv in self.kv]
        self.bwd_bufs = [[[torch.empty_like(t) for t in self.kv[r] + self.dkv[r]]
                          for _ in range(2)] for r in range(P)]

    def bwd(self):
        P = self.P
        cur = [self.kv[r] + self.dkv[r] for r in range(P)]
        self._run(self.bwd_ranks, cur, self.bwd_bufs, range(4))
        # rank r holds the finished dK/dV of rank (r + 1) mod P
        return ([rk.dq for rk in self.bwd_ranks], [cur[(r - 1) % P][2] for r in range(P)],
                [cur[(r - 1) % P][3] for r in range(P)])


def emulate_ring_fwd(q, k, v, *, num_shards, layout, causal, cu_seqlens=None):
    """The multi-GPU ring forward with all P ranks on this GPU (EmulatedRing).
    q, k, v are whole-sequence tensors; returns whole-sequence (out, lse)
    gathered from the ranks."""
    ring = EmulatedRing(q, k, v, num_shards=num_shards, layout=layout, causal=causal,
                        cu_seqlens=cu_seqlens)
    outs, lses = zip(*ring.fwd())
    return unshard(outs, num_shards, layout), unshard(lses, num_shards, layout, dim=1)


def _emulated_pass_on(cur, bufs, s, streams, computed, fields):
    """Rank r copies fields of cur[r] into rank r+1's receive buffer s % 2, on
    its own stream, once rank r+1 has finished step s (which frees that
    buffer); then every rank's next step waits for its copy to arrive."""
    import torch
    P = len(cur)
    arrived = [torch.cuda.Event() for _ in range(P)]
    for r in range(P):
        dst = (r + 1) % P
        st = streams[r]
        st.wait_event(computed[dst])
        with torch.cuda.stream(st):
            for f in fields:
                bufs[dst][s % 2][f].copy_(cur[r][f], non_blocking=True)
            arrived[dst].record(st)
    for r in range(P):
        streams[r].wait_event(arrived[r])
        for f in fields:
            cur[r][f] = bufs[r][s % 2][f]


def emulate_ring_bwd(q, k, v, out, lse, dout, *, num_shards, layout, causal, cu_seqlens=None):
    """The multi-GPU ring backward with all P ranks on this GPU (EmulatedRing).
    out and lse are whole-sequence forward results.  Returns whole-sequence
    fp32 (dq, dk, dv)."""
    ring = EmulatedRing(q, k, v, num_shards=num_shards, layout=layout, causal=causal,
                        cu_seqlens=cu_seqlens)
    ring.prepare_bwd(out, lse, dout)
    dqs, dks, dvs = ring.bwd()
    return (unshard(dqs, num_shards, layout), unshard(dks, num_shards, layout),
            unshard(dvs, num_shards, layout))
