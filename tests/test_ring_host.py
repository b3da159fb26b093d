"""The multi-GPU ring's host side, run as gloo ranks on the CPU.

The ring driver (context_long_sequence_fwd_b300/ring.py) passes K/V shards
from rank to rank (aicassindra "tm_sp_math", "Context parallelism is the axis
that is independent": K/V blocks rotate around a ring) and folds each step
into the rank's running result (axolotl "Sequence Parallelism" page,
introduction: results aggregated through a ring).  Here each rank is a
process talking gloo, and the per-step computation is replaced by stand-ins
built on the oracle:

* forward: each step computes the partial attention of the rank's rows over
  exactly the keys of the shard the schedule says it holds (the oracle with
  those keys allowed), from the K/V rows it actually received, and merges it
  into the running result with the oracle's log-sum-exp merge.  Every rank's
  rows must equal the oracle's whole-sequence attention: a shard delivered to
  the wrong rank, at the wrong step, twice or never, breaks that.
* backward: each step checks that the K/V it holds are the scheduled shard's
  rows, adds a tag naming (rank, shard) to dq and to the shard's travelling
  dK/dV accumulators; afterwards dq holds one tag per shard and every owner
  got back its own dK/dV with one tag per rank.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from context_long_sequence_fwd_b300 import CONTIGUOUS, ZIGZAG
from context_long_sequence_fwd_b300 import ring


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def problem(T, hq, hkv, d, seed):
    r = np.random.default_rng(seed)
    return tuple(torch.from_numpy(r.standard_normal(s)) for s in
                 ((T, hq, d), (T, hkv, d), (T, hkv, d), (T, hq, d)))


def token_index(T, P, layout, rank):
    return np.concatenate([np.arange(a, b) for a, b in ring.rank_rows(T, P, layout, rank)])


class OracleFwdRank:
    """Forward step stand-in: the oracle's partial attention of this rank's
    rows over the keys of the shard held at this step, merged step by step."""

    def __init__(self, q_full, T, P, layout, causal, rank, cu):
        self.q_full, self.T, self.P, self.layout = q_full, T, P, layout
        self.causal, self.rank, self.cu = causal, rank, cu
        self.rows = token_index(T, P, layout, rank)
        self.o = self.lse = None

    def __call__(self, step, k, v):
        src = (self.rank - step) % self.P
        keys = token_index(self.T, self.P, self.layout, src)
        hq, hkv, d = self.q_full.shape[1], k.shape[1], k.shape[2]
        kg = np.zeros((self.T, hkv, d))
        vg = np.zeros((self.T, hkv, d))
        kg[keys], vg[keys] = k.numpy(), v.numpy()   # the rows this rank received
        allowed = np.zeros(self.T, bool)
        allowed[keys] = True
        hs = np.repeat(np.arange(hq, dtype=np.int32), self.rows.size)
        is_ = np.tile(self.rows.astype(np.int32), hq)
        o, lse = oracle.fwd_rows(self.q_full, kg, vg, hs, is_, causal=self.causal,
                                 cu_seqlens=self.cu, key_allowed=allowed)
        if self.o is None:
            self.o, self.lse = o, lse
        else:
            self.o, self.lse = oracle.lse_merge(self.o, self.lse, o, lse)

    def result(self):
        hq = self.q_full.shape[1]
        n = self.rows.size
        return self.o.reshape(hq, n, -1).transpose(1, 0, 2), self.lse.reshape(hq, n)


class TagBwdRank:
    """Backward step stand-in: checks the K/V it holds and adds tags."""

    def __init__(self, k_full, T, P, layout, rank, q_rows):
        self.k_full, self.T, self.P, self.layout, self.rank = k_full, T, P, layout, rank
        self.dq = torch.zeros(q_rows.shape, dtype=torch.float64)
        self.steps = []

    def __call__(self, step, k, v, dk, dv):
        src = (self.rank - step) % self.P
        assert torch.equal(k, ring.shard(self.k_full, self.P, self.layout, src))
        self.steps.append(src)
        self.dq += 1000.0 ** src
        tag = 1000.0 ** self.rank
        if step == 0:   # the shard's owner starts its accumulators
            dk.fill_(tag)
            dv.fill_(-tag)
        else:
            dk += tag
            dv -= tag


def _worker(rank, world, port, case, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        T, hq, hkv, d, layout, causal, cu = case
        q, k, v, do = problem(T, hq, hkv, d, seed=5)
        qs, ks, vs = (ring.shard(t, world, layout, rank) for t in (q, k, v))
        step = OracleFwdRank(q.numpy(), T, world, layout, causal, rank, cu)
        o, lse = ring.ring_fwd(qs, ks, vs, total_tokens=T, layout=layout, causal=causal,
                               cu_seqlens=cu, rank_step=step)
        tag = TagBwdRank(k, T, world, layout, rank, qs)
        dq, dk, dv = ring.ring_bwd(qs, ks, vs, qs, None, qs, total_tokens=T, layout=layout,
                                   causal=causal, cu_seqlens=cu, rank_step=tag)
        out_q.put((rank, o, lse, tag.steps, dq.numpy(), dk.numpy(), dv.numpy()))
    finally:
        dist.destroy_process_group()


CASES = [
    # T, hq, hkv, d, layout, causal, cu_seqlens
    (48, 4, 2, 8, ZIGZAG, True, None),
    (40, 2, 1, 4, CONTIGUOUS, True, [0, 7, 8, 30, 40]),
    (32, 2, 2, 4, CONTIGUOUS, False, [0, 12, 32]),
]


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("case", CASES, ids=str)
def test_ring_schedule_gloo(case, world):
    T, hq, hkv, d, layout, causal, cu = case
    if T % (world * (2 if layout == ZIGZAG else 1)):
        T = T // (2 * world) * 2 * world
        cu = None if cu is None else [min(c, T) for c in cu[:-1]] + [T]
        case = (T, hq, hkv, d, layout, causal, cu)
    ctx = mp.get_context("spawn")
    out_q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, case, out_q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in procs:
        r, *res = out_q.get(timeout=180)
        got[r] = res
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    q, k, v, _ = problem(T, hq, hkv, d, seed=5)
    ref_o, ref_l = oracle.attention_fwd(q.numpy(), k.numpy(), v.numpy(), causal=causal,
                                        cu_seqlens=cu)
    for r in range(world):
        o, lse, steps, dq, dk, dv = got[r]
        rows = token_index(T, world, layout, r)
        assert np.max(np.abs(o - ref_o[rows])) < 1e-12
        assert np.max(np.abs(lse - ref_l[:, rows])) < 1e-12
        # the ring visits every shard once, in ring order
        assert steps == [(r - s) % world for s in range(world)]
        assert np.all(dq == sum(1000.0 ** s for s in range(world)))
        # the owner's keys got one tag from every rank, and came back home
        assert np.all(dk == sum(1000.0 ** x for x in range(world)))
        assert np.all(dv == -sum(1000.0 ** x for x in range(world)))


def test_shard_and_unshard_are_inverse():
    x = torch.arange(48 * 3).reshape(48, 3)
    for layout in (CONTIGUOUS, ZIGZAG):
        for P in (1, 2, 3, 4):
            if 48 % (2 * P if layout == ZIGZAG else P):
                continue
            parts = [ring.shard(x, P, layout, r) for r in range(P)]
            assert sum(p.shape[0] for p in parts) == 48
            assert torch.equal(ring.unshard(parts, P, layout), x)
            if layout == ZIGZAG:
                C = 48 // (2 * P)
                assert torch.equal(parts[0][:C], x[:C]) and torch.equal(parts[0][C:], x[-C:])
