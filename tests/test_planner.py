"""Host-side checks of the shard / ring-step planner (no GPU).

The planner's work list must cover, for every query row and head, exactly the
keys the causal / document mask lets it see -- no key missing, none visited
twice -- visit them in ring order (step s reads the K/V shard of rank
(r - s) mod P, axolotl "Sequence Parallelism" page, introduction), skip key
ranges nobody can see (causal skip), and keep ZIGZAG's per-rank causal work
equal (aicassindra "tm_sp_math", "Context parallelism is the axis that is
independent": the causal-mask load-balance problem).
"""
import numpy as np
import pytest

import context_long_sequence_fwd_b300 as ra
from context_long_sequence_fwd_b300.workloads import cu_seqlens_from_lengths, doc_lengths

TILE = 128


def doc_index(T, cu):
    bounds = [0, T] if cu is None else [int(x) for x in cu]
    doc = np.empty(T, np.int64)
    for d, (a, b) in enumerate(zip(bounds[:-1], bounds[1:])):
        doc[a:b] = d
    return doc


def visible_keys(i, doc, causal):
    ks = np.nonzero(doc == doc[i])[0]
    return ks[ks <= i] if causal else ks


def rank_chunks(T, P, layout, r):
    if layout == ra.CONTIGUOUS:
        C = T // P
        return [(r * C, (r + 1) * C)]
    C = T // (2 * P)
    return [(r * C, (r + 1) * C), ((2 * P - 1 - r) * C, (2 * P - r) * C)]


CASES = [
    # T, hq, hkv, P, layout, causal, cu
    (512, 2, 2, 2, ra.CONTIGUOUS, True, None),
    (512, 4, 2, 4, ra.ZIGZAG, True, None),
    (768, 2, 1, 3, ra.CONTIGUOUS, False, None),
    (1000, 2, 2, 2, ra.CONTIGUOUS, True, None),        # chunks of 500: ragged tiles
    (1040, 4, 2, 4, ra.ZIGZAG, True, None),            # zigzag chunks of 130
    (1024, 4, 1, 4, ra.CONTIGUOUS, True, [0, 100, 101, 400, 777, 1024]),
    (960, 6, 2, 2, ra.CONTIGUOUS, False, [0, 300, 310, 960]),
    (1024, 2, 2, 2, ra.ZIGZAG, True, [0, 200, 200, 900, 1024]),   # empty document
    (256, 3, 3, 1, ra.CONTIGUOUS, True, None),         # P = 1
    (384, 2, 2, 1, ra.ZIGZAG, True, None),             # zigzag with one rank
]


def check_plan(T, hq, hkv, P, layout, causal, cu, hks=1, exchange=ra.RING):
    items, segs = ra.plan_fwd(T, hq, hkv, P, layout, causal, cu, heads_k_stride=hks,
                              kv_exchange=exchange)
    doc = doc_index(T, cu)
    G = hq // hkv
    seen = np.zeros((hq, T), np.int64)
    for it in items:
        (q0a, q0b, qla, qlb, ha, hb, sb, sc, rank, cost, mla, mlb, mha, mhb, pas, _) = it
        my = segs[sb:sb + sc]
        if exchange == ra.ALLGATHER:
            # gathered K/V: at most one range, in token order, in step 0
            assert sc <= 1 and np.all(my[:, 2] == 0) and np.all(my[:, 3] == -1)
        else:
            # ring order and shard ownership of every segment
            assert np.all(np.diff(my[:, 2]) >= 0), "segments out of ring order"
        for k0, k1, step, src in my:
            assert k0 < k1
            if exchange == ra.RING:
                assert src == (rank - step) % P
                assert any(a <= k0 and k1 <= b for a, b in rank_chunks(T, P, layout, src))
        keys = np.concatenate([np.arange(k0, k1) for k0, k1, _, _ in my]) if len(my) else \
            np.zeros(0, np.int64)
        assert len(np.unique(keys)) == len(keys), "a key is visited twice"
        assert cost == sum((k1 - k0 + TILE - 1) // TILE for k0, k1, _, _ in my)
        rows_all = []
        for q0, ql, h, mlo, mhi in ((q0a, qla, ha, mla, mha), (q0b, qlb, hb, mlb, mhb)):
            if ql == 0:
                continue
            assert h // G == ha // G, "tiles of an item share a kv head"
            assert pas == (h // G) // hks
            assert any(a <= q0 and q0 + ql <= b for a, b in rank_chunks(T, P, layout, rank))
            rows = np.arange(q0, q0 + ql)
            rows_all.append(rows)
            seen[h, rows] += 1
            for i in rows:
                vis = visible_keys(i, doc, causal)
                got = np.intersect1d(keys, vis)
                assert len(got) == len(vis), f"row {i} misses keys"
            # a tile inside [mask_lo, mask_hi) needs no mask: every key of it
            # must be visible to every row of the query tile
            lo_i = np.array([visible_keys(i, doc, causal).min() for i in rows])
            hi_i = np.array([visible_keys(i, doc, causal).max() + 1 for i in rows])
            assert mlo == lo_i.max() and mhi == hi_i.min()
        # causal skip is tight: every visited key is visible to some row
        rows_all = np.concatenate(rows_all)
        vis_any = np.zeros(T, bool)
        for i in rows_all:
            vis_any[visible_keys(i, doc, causal)] = True
        assert np.all(vis_any[keys]), "a segment holds keys no row can see"
    assert np.all(seen == 1), "every (head, row) belongs to exactly one tile"
    # longest first inside each pass
    for p in np.unique(items[:, 14]):
        c = items[items[:, 14] == p, 9]
        assert np.all(np.diff(c) <= 0)
    passes = items[:, 14]
    assert np.all(np.diff(passes) >= 0), "passes run in order"
    return items, segs


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_plan_covers_exactly_the_mask(case):
    check_plan(*case)


@pytest.mark.parametrize("hks", [1, 2, 4])
def test_heads_k_stride_groups_passes(hks):
    items, _ = check_plan(512, 8, 4, 2, ra.ZIGZAG, True, None, hks=hks)
    assert items[:, 14].max() == 4 // hks - 1


def test_zigzag_balances_causal_work():
    T, P = 4096, 4
    items, segs = ra.plan_fwd(T, 1, 1, P, ra.ZIGZAG, True)
    pairs = np.zeros(P)
    step_pairs = np.zeros((P, P))
    for it in items:
        for q0, ql in ((it[0], it[2]), (it[1], it[3])):
            if ql == 0:
                continue
            for k0, k1, step, src in segs[it[6]:it[6] + it[7]]:
                # visible (q, k) pairs of this tile and segment
                qi = np.arange(q0, q0 + ql)[:, None]
                kj = np.arange(k0, k1)[None, :]
                n = int(np.sum(kj <= qi))
                pairs[it[8]] += n
                step_pairs[it[8], step] += n
    assert np.all(pairs == pairs[0]), pairs
    C = T // (2 * P)
    for r in range(P):
        for s in range(1, P):
            # every non-diagonal step is exactly half of a 2C x 2C block
            assert step_pairs[r, s] == 2 * C * C


def test_contiguous_causal_skips_future_shards():
    T, P = 2048, 4
    items, segs = ra.plan_fwd(T, 1, 1, P, ra.CONTIGUOUS, True)
    for it in items:
        r = it[8]
        srcs = set(segs[it[6]:it[6] + it[7], 3])
        assert all(s <= r for s in srcs)          # shards after r are never visited


def test_varlen_workload_plan():
    lens = doc_lengths(65536, 512, 8192, 1)
    cu = cu_seqlens_from_lengths(lens).numpy()
    assert cu[-1] == 65536 and all(512 <= x <= 8192 for x in lens[:-1])
    items, segs = ra.plan_fwd(65536, 32, 8, 8, ra.CONTIGUOUS, True, cu)
    # every segment stays inside one document of the item's first row
    doc = doc_index(65536, cu)
    for it in items[:200]:
        for k0, k1, _, _ in segs[it[6]:it[6] + it[7]]:
            assert doc[k0] >= doc[it[0]]


@pytest.mark.parametrize("T,P,layout", [(1000, 3, ra.CONTIGUOUS), (1000, 3, ra.ZIGZAG),
                                        (512, 3, ra.ZIGZAG)])
def test_not_divisible_is_rejected(T, P, layout):
    with pytest.raises(ra.RingAttnError) as e:
        ra.plan_fwd(T, 2, 2, P, layout, True)
    assert e.value.code == -2


@pytest.mark.parametrize("cu", [[0, 10, 9, 100], [1, 100], [0, 50], [0]])
def test_bad_cu_seqlens_rejected(cu):
    with pytest.raises(ra.RingAttnError) as e:
        ra.plan_fwd(100, 2, 2, 1, ra.CONTIGUOUS, True, np.array(cu, np.int32))
    assert e.value.code == -1


def test_empty_sequence_plan():
    items, segs = ra.plan_fwd(0, 2, 2, 2, ra.CONTIGUOUS, True)
    assert len(items) == 0 and len(segs) == 0


def check_bwd_plan(T, hq, hkv, P, layout, causal, cu, hks=1):
    items, segs = ra.plan_bwd(T, hq, hkv, P, layout, causal, cu, heads_k_stride=hks)
    doc = doc_index(T, cu)
    seen = np.zeros((hkv, T), np.int64)
    for k0, klen, g, src, sb, sc, cost, _ in items:
        assert 1 <= klen <= TILE
        assert any(a <= k0 and k0 + klen <= b for a, b in rank_chunks(T, P, layout, src))
        seen[g, k0:k0 + klen] += 1
        my = segs[sb:sb + sc]
        # the whole-GPU plan walks the query segments from the sequence's end
        # down (L2 reuse); every segment keeps its ring step and rank
        assert np.all(np.diff(my[:, 0]) < 0), "segments not in descending query order"
        for q0, q1, step, rank in my:
            assert rank == (src + step) % P
            assert any(a <= q0 and q1 <= b for a, b in rank_chunks(T, P, layout, rank))
        rows = np.concatenate([np.arange(q0, q1) for q0, q1, _, _ in my])
        assert len(np.unique(rows)) == len(rows), "a query row is visited twice"
        assert cost == sum((q1 - q0 + TILE - 1) // TILE for q0, q1, _, _ in my) * (hq // hkv)
        # every query that sees a key of the tile is visited, and no other
        need = np.zeros(T, bool)
        for j in range(k0, k0 + klen):
            for i in range(T):
                if doc[i] == doc[j] and (not causal or j <= i):
                    need[i] = True
        got = np.zeros(T, bool)
        got[rows] = True
        assert np.array_equal(need, got)
    assert np.all(seen == 1), "every key of every kv head in exactly one tile"


@pytest.mark.parametrize("case", CASES[:8], ids=[str(i) for i in range(8)])
def test_bwd_plan_covers_exactly_the_mask(case):
    check_bwd_plan(*case)


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_allgather_plan_covers_exactly_the_mask(case):
    """The all-gather exchange (varlen_llama3) visits the same keys as the
    ring, in token order."""
    T, hq, hkv, P, layout, causal, cu = case
    items, segs = check_plan(T, hq, hkv, P, layout, causal, cu, exchange=ra.ALLGATHER)
    ring_items, _ = check_plan(T, hq, hkv, P, layout, causal, cu)
    # the same query tiles; gathered keys are one range, so whole tiles can
    # span shard boundaries and an item never visits more K/V tiles
    key = lambda a: sorted(map(tuple, a[:, [0, 1, 2, 3, 4, 5]].tolist()))
    assert key(items) == key(ring_items)
    assert items[:, 9].sum() <= ring_items[:, 9].sum()


def test_allgather_bwd_plan_covers_exactly_the_mask():
    for case in CASES[:8]:
        T, hq, hkv, P, layout, causal, cu = case
        items, segs = ra.plan_bwd(T, hq, hkv, P, layout, causal, cu, kv_exchange=ra.ALLGATHER)
        ring, _ = ra.plan_bwd(T, hq, hkv, P, layout, causal, cu)
        assert items[:, 6].sum() <= ring[:, 6].sum()  # never more work than the ring
        doc = doc_index(T, cu)
        for k0, klen, g, src, sb, sc, cost, _ in items:
            assert sc <= 1
            for q0, q1, step, rank in segs[sb:sb + sc]:
                assert step == 0 and rank == -1
                # exactly the queries that see some key of the tile
                want = [i for i in range(T)
                        if any(np.isin(np.arange(k0, k0 + klen), visible_keys(i, doc, causal)))]
                assert list(range(q0, q1)) == want


# ------------------------------------------- the fused forward's work list

def item_keys(items, segs):
    """(query tiles) -> keys visited, concatenated over every item on them."""
    out = {}
    for it in items:
        key = (int(it[0]), int(it[2]), int(it[4]), int(it[1]), int(it[3]), int(it[5]))
        my = segs[it[6]:it[6] + it[7]]
        ks = [np.arange(k0, k1) for k0, k1, _, _ in my]
        out.setdefault(key, []).extend(ks)
    return {k: np.sort(np.concatenate(v)) if v else np.zeros(0, np.int64) for k, v in out.items()}


def claim_makespan(costs, sms):
    """Finish time of the last CTA when sms CTAs claim items in list order."""
    import heapq
    h = [0] * sms
    for c in costs:
        heapq.heappush(h, heapq.heappop(h) + c)
    return max(h)


FUSED_CASES = CASES + [
    (8192, 8, 8, 4, ra.ZIGZAG, True, None),              # the causal MHA workload at 8K
    (2048, 4, 2, 4, ra.ZIGZAG, True, [0, 300, 301, 900, 2048]),
]


@pytest.mark.parametrize("sms", [148, 7])
@pytest.mark.parametrize("case", FUSED_CASES, ids=[str(i) for i in range(len(FUSED_CASES))])
def test_fused_list_covers_the_plan(case, sms):
    """The fused forward's list (claim order, long items split in two) visits
    exactly the plan's keys for every pair of query tiles, each once; split
    halves cover the first and second half of the item's key tiles in ring
    order; items run longest first inside each ordering group."""
    T, hq, hkv, P, layout, causal, cu = case
    items, segs = ra.plan_fwd(T, hq, hkv, P, layout, causal, cu)
    fi, fs = ra.plan_fwd_fused(T, hq, hkv, P, layout, causal, sms, cu)
    ref, got = item_keys(items, segs), item_keys(fi, fs)
    assert ref.keys() == got.keys()
    for k in ref:
        assert np.array_equal(np.sort(ref[k]), got[k]), k
        assert len(np.unique(got[k])) == len(got[k])
    mean = items[:, 9].sum() / sms
    parts = fi[:, 15]
    assert np.all(items[:, 15] == -1)
    for it in fi:
        my = fs[it[6]:it[6] + it[7]]
        assert it[9] == sum((k1 - k0 + TILE - 1) // TILE for k0, k1, _, _ in my)
        assert np.all(np.diff(my[:, 2]) >= 0), "ring order inside an item"
    # split items: halves 2 i and 2 i + 1 of one item longer than the mean
    n_pairs = (parts >= 0).sum() // 2
    assert sorted(parts[parts >= 0]) == list(range(2 * n_pairs))
    by_part = {int(it[15]): it for it in fi if it[15] >= 0}
    for i in range(n_pairs):
        a, b = by_part[2 * i], by_part[2 * i + 1]
        assert np.array_equal(a[:6], b[:6]), "halves share the query tiles"
        total = a[9] + b[9]
        assert total > mean and a[9] == (total + 1) // 2
        ka = np.concatenate([np.arange(k0, k1) for k0, k1, _, _ in fs[a[6]:a[6] + a[7]]])
        kb = np.concatenate([np.arange(k0, k1) for k0, k1, _, _ in fs[b[6]:b[6] + b[7]]])
        sa = fs[a[6]:a[6] + a[7]]
        sb = fs[b[6]:b[6] + b[7]]
        assert (sa[-1, 2], sa[-1, 1]) <= (sb[0, 2], sb[0, 0]), "first half comes first in the ring"
        assert len(np.intersect1d(ka, kb)) == 0
    for it in fi[parts < 0]:
        assert it[9] <= mean or it[9] < 2
    # the claim order balances at least as well as the plan order
    assert claim_makespan(fi[:, 9], sms) <= claim_makespan(items[:, 9], sms)


def test_fused_list_balances_the_8k_workload():
    """The causal MHA workload at 8K (256 items of up to 64 key tiles for
    148 SMs): claiming the plan in pass order leaves the last CTAs with about
    94 tiles against a mean of 57; the fused list brings it within 10 %."""
    T, hq, hkv, P = 8192, 8, 8, 4
    items, _ = ra.plan_fwd(T, hq, hkv, P, ra.ZIGZAG, True)
    fi, _ = ra.plan_fwd_fused(T, hq, hkv, P, ra.ZIGZAG, True, 148)
    mean = items[:, 9].sum() / 148
    assert claim_makespan(items[:, 9], 148) > 1.5 * mean
    assert claim_makespan(fi[:, 9], 148) <= 1.1 * mean


def test_fused_list_of_a_big_problem_keeps_pass_order():
    """At 32K tokens every pass over a key/value head has more than 2 x 148
    items: the fused list keeps one pass per ordering group (K/V of few heads
    in flight) and splits nothing."""
    items, _ = ra.plan_fwd(32768, 32, 8, 8, ra.ZIGZAG, True)
    fi, _ = ra.plan_fwd_fused(32768, 32, 8, 8, ra.ZIGZAG, True, 148)
    assert len(fi) == len(items) and np.all(fi[:, 15] == -1)
    assert np.all(np.diff(fi[:, 14]) >= 0)


def test_plans_past_2_31_elements_cover_the_causal_mask():
    """786432 tokens, 32 / 8 heads, 8 zigzag shards (q holds 3.2e9 values):
    every forward item's key segments tile [0, end of its rows) exactly once,
    and every backward key tile's query segments tile [its first key, T)
    exactly once, so the plans stay exact where the tensors pass 2^31
    elements."""
    T, hq, hkv, P = 786432, 32, 8, 8
    items, segs = ra.plan_fwd(T, hq, hkv, P, ra.ZIGZAG, True)
    assert len(items) == (T // TILE) * hq // 2
    for it in items:
        s = segs[it[6]:it[6] + it[7]]
        s = s[np.argsort(s[:, 0])]
        end = max(it[0] + it[2], it[1] + it[3])
        assert s[0, 0] == 0 and s[-1, 1] == end and np.all(s[1:, 0] == s[:-1, 1])
    bitems, bsegs = ra.plan_bwd(T, hq, hkv, P, ra.ZIGZAG, True)
    assert len(bitems) == (T // TILE) * hkv
    for k0, klen, g, src, sb, sc, cost, _ in bitems:
        s = bsegs[sb:sb + sc]
        s = s[np.argsort(s[:, 0])]
        assert s[0, 0] == k0 and s[-1, 1] == T and np.all(s[1:, 0] == s[:-1, 1])
        assert cost == (T - k0) // TILE * (hq // hkv)
