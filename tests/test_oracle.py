"""Pins for the fp64 oracle: it is checked against things other than itself.

* brute force on tiny inputs: the full score matrix built with numpy, an
  explicit mask matrix built from the definition of the visible set, and
  scipy's softmax / logsumexp;
* closed forms: q = 0 gives the mean of the visible values and ln|V(i)|; a row
  that sees one key returns that key's value; a dominant score picks its value;
  a D = 1, T = 2 case worked by hand;
* invariants: v = 1 gives O = 1 (softmax rows sum to one); the log-sum-exp
  merge of any partition of the keys (random, or the ring's contiguous and
  zigzag chunks in ring order) equals the unpartitioned result; the merge
  itself equals numpy's logaddexp; D_i = dO_i . O_i; sum_j dK_j = 0 and
  sum_j dV_j = sum over the group's queries of dO;
* finite differences of L = sum(dO * O) against the analytic gradients.

The pins that speak only of the definition take the implementation as an
argument, so the same checks also pin the matrix-product oracle
(``oracle.blas``, see test_oracle_blas.py).

These follow the definition of attention the ring schedule must reproduce
(every query sees every key of its document, axolotl "Sequence Parallelism"
page, introduction; aicassindra "tm_sp_math", "Context parallelism is the axis
that is independent"; positions reset per packed sample, "Sample Packing with
Sequence Parallelism").
"""
import math

import numpy as np
import pytest
import scipy.special

import oracle

# ----------------------------------------------------------------- helpers


def rand_qkv(T, hq, hkv, d, seed, with_do=True):
    r = np.random.default_rng(seed)
    q = r.standard_normal((T, hq, d))
    k = r.standard_normal((T, hkv, d))
    v = r.standard_normal((T, hkv, d))
    do = r.standard_normal((T, hq, d))
    return (q, k, v, do) if with_do else (q, k, v)


def mask_matrix(T, cu, causal):
    """Explicit [T, T] visibility matrix, enumerated document by document."""
    M = np.zeros((T, T), bool)
    bounds = [0, T] if cu is None else list(cu)
    for a, b in zip(bounds[:-1], bounds[1:]):
        for i in range(a, b):
            for j in range(a, b):
                if not causal or j <= i:
                    M[i, j] = True
    return M


def brute_force(q, k, v, cu, causal, scale=None):
    T, hq, d = q.shape
    hkv = k.shape[1]
    G = hq // hkv
    sc = 1.0 / math.sqrt(d) if scale is None else scale
    M = mask_matrix(T, cu, causal)
    O = np.zeros_like(q)
    L = np.zeros((hq, T))
    for h in range(hq):
        g = h // G
        S = sc * (q[:, h, :] @ k[:, g, :].T)
        Sm = np.where(M, S, -np.inf)
        L[h] = scipy.special.logsumexp(Sm, axis=1)
        O[:, h, :] = scipy.special.softmax(Sm, axis=1) @ v[:, g, :]
    return O, L


CASES = [
    # T, hq, hkv, d, cu_seqlens, causal
    (48, 4, 2, 8, None, True),
    (40, 2, 2, 16, None, False),
    (64, 6, 2, 8, [0, 10, 11, 30, 64], True),
    (64, 3, 1, 4, [0, 7, 40, 64], False),
    (33, 4, 4, 5, [0, 1, 2, 20, 33], True),
    (30, 2, 1, 4, [0, 0, 10, 10, 30], True),          # empty documents
]


# ------------------------------------------------------------ pin checks
# Written as functions so the mutation tests can run them on a broken oracle.

def check_bruteforce(seed=0, impl=oracle):
    for (T, hq, hkv, d, cu, causal) in CASES:
        q, k, v = rand_qkv(T, hq, hkv, d, seed, with_do=False)
        o, lse = impl.attention_fwd(q, k, v, causal=causal, cu_seqlens=cu)
        ob, lb = brute_force(q, k, v, cu, causal)
        assert np.max(np.abs(o - ob)) < 1e-12
        assert np.max(np.abs(lse - lb)) < 1e-12


def check_fd_gradients(impl=oracle):
    T, hq, hkv, d = 12, 4, 2, 3
    cu = [0, 5, 12]
    q, k, v, do = rand_qkv(T, hq, hkv, d, 7)

    def loss(q_, k_, v_):
        o, _ = impl.attention_fwd(q_, k_, v_, causal=True, cu_seqlens=cu)
        return float(np.sum(do * o))

    dq, dk, dv, _, _ = impl.attention_bwd(q, k, v, do, causal=True, cu_seqlens=cu)
    h = 1e-5
    r = np.random.default_rng(3)
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(12):
            idx = tuple(int(r.integers(0, n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd = (loss(**{a + "_": b for a, b in args_p.items()})
                  - loss(**{a + "_": b for a, b in args_m.items()})) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, g[idx])


def check_partition_merge(impl=oracle):
    T, hq, hkv, d = 64, 4, 2, 8
    cu = [0, 9, 41, 64]
    q, k, v = rand_qkv(T, hq, hkv, d, 11, with_do=False)
    o_full, l_full = impl.attention_fwd(q, k, v, causal=True, cu_seqlens=cu)
    r = np.random.default_rng(5)
    partitions = []
    labels = r.integers(0, 3, T)                       # random 3-way partition
    partitions.append([labels == p for p in range(3)])
    P = 4                                              # contiguous ring chunks
    C = T // P
    partitions.append([np.arange(T) // C == p for p in range(P)])
    C2 = T // (2 * P)                                  # zigzag: chunks r, 2P-1-r
    chunk = np.arange(T) // C2
    partitions.append([(chunk == p) | (chunk == 2 * P - 1 - p) for p in range(P)])
    for parts in partitions:
        order = r.permutation(len(parts))
        acc_o, acc_l = None, None
        for p in order:
            o_p, l_p = impl.attention_fwd(q, k, v, causal=True, cu_seqlens=cu,
                                          key_allowed=parts[p])
            o_p = o_p.transpose(1, 0, 2)               # [Hq, T, D] rows match lse
            if acc_o is None:
                acc_o, acc_l = o_p, l_p
            else:
                acc_o, acc_l = oracle.lse_merge(acc_o, acc_l, o_p, l_p)
        assert np.max(np.abs(acc_o.transpose(1, 0, 2) - o_full)) < 1e-12
        assert np.max(np.abs(acc_l - l_full)) < 1e-12


def check_merge_rule():
    r = np.random.default_rng(1)
    n, d = 50, 6
    oa, ob = r.standard_normal((n, d)), r.standard_normal((n, d))
    la, lb = r.standard_normal(n) * 5, r.standard_normal(n) * 5
    la[3] = -np.inf
    lb[4] = -np.inf
    la[5] = lb[5] = -np.inf
    oa[5] = ob[5] = 0.0
    om, lm = oracle.lse_merge(oa, la, ob, lb)
    ref_l = np.logaddexp(la, lb)
    assert np.array_equal(np.isinf(lm), np.isinf(ref_l))
    fin = np.isfinite(ref_l)
    assert np.max(np.abs(lm[fin] - ref_l[fin])) < 1e-13
    wa = np.where(np.isfinite(la), np.exp(la - np.where(fin, ref_l, 0)), 0.0)
    wb = np.where(np.isfinite(lb), np.exp(lb - np.where(fin, ref_l, 0)), 0.0)
    ref_o = wa[:, None] * oa + wb[:, None] * ob
    assert np.max(np.abs(om - ref_o)) < 1e-13
    assert np.array_equal(om[3], ob[3]) and np.array_equal(om[4], oa[4])
    assert np.all(om[5] == 0.0) and lm[5] == -np.inf


def check_backward_identities(impl=oracle):
    T, hq, hkv, d = 40, 6, 2, 8
    cu = [0, 13, 40]
    q, k, v, do = rand_qkv(T, hq, hkv, d, 21)
    o, lse = impl.attention_fwd(q, k, v, causal=True, cu_seqlens=cu)
    dq, dk, dv, D, l2 = impl.attention_bwd(q, k, v, do, causal=True, cu_seqlens=cu)
    assert np.max(np.abs(l2 - lse)) < 1e-12
    # D_i = sum_j P_ij dP_ij equals dO_i . O_i
    assert np.max(np.abs(D - np.einsum("thd,thd->ht", do, o))) < 1e-12
    G = hq // hkv
    for g in range(hkv):
        # rows of dS sum to zero, so the keys' dK sum to zero
        assert np.max(np.abs(dk[:, g, :].sum(0))) < 1e-12
        # rows of P sum to one, so the keys' dV sum to the group's dO
        ref = do[:, g * G:(g + 1) * G, :].sum((0, 1))
        assert np.max(np.abs(dv[:, g, :].sum(0) - ref)) < 1e-11


def check_closed_forms(impl=oracle):
    T, hq, hkv, d = 30, 2, 1, 4
    cu = [0, 12, 30]
    _, k, v = rand_qkv(T, hq, hkv, d, 2, with_do=False)
    q = np.zeros((T, hq, d))
    M = mask_matrix(T, cu, True)
    o, lse = impl.attention_fwd(q, k, v, causal=True, cu_seqlens=cu)
    for i in range(T):
        vis = np.nonzero(M[i])[0]
        for h in range(hq):
            assert abs(lse[h, i] - math.log(len(vis))) < 1e-13
            assert np.max(np.abs(o[i, h] - v[vis, 0].mean(0))) < 1e-13
    # the first row of each document sees only itself
    q2, k2, v2 = rand_qkv(T, hq, hkv, d, 3, with_do=False)
    o2, l2 = impl.attention_fwd(q2, k2, v2, causal=True, cu_seqlens=cu)
    for i in cu[:-1]:
        for h in range(hq):
            assert np.max(np.abs(o2[i, h] - v2[i, 0])) < 1e-13
            s = float(q2[i, h] @ k2[i, 0]) / math.sqrt(d)
            assert abs(l2[h, i] - s) < 1e-13
    # v = 1 everywhere: every row's weights sum to one, so O = 1
    o3, _ = impl.attention_fwd(q2, k2, np.ones_like(v2), causal=False)
    assert np.max(np.abs(o3 - 1.0)) < 1e-13


def check_dominant_key(impl=oracle):
    T, d = 16, 4
    r = np.random.default_rng(9)
    q = r.standard_normal((T, 1, d)) * 0.01
    k = r.standard_normal((T, 1, d)) * 0.01
    v = r.standard_normal((T, 1, d))
    q[:, 0, :] += np.array([1.0, 0, 0, 0]) * 60.0
    k[5, 0, :] = np.array([1.0, 0, 0, 0]) * 60.0   # score 1800 for key 5
    o, _ = impl.attention_fwd(q, k, v, causal=False)
    assert np.max(np.abs(o[:, 0, :] - v[5, 0])) < 1e-12


def check_hand_case(impl=oracle):
    # D = 1, T = 2, non-causal, scale 1: q = (1, 2), k = (0.5, -1), v = (3, 5)
    q = np.array([[[1.0]], [[2.0]]])
    k = np.array([[[0.5]], [[-1.0]]])
    v = np.array([[[3.0]], [[5.0]]])
    o, lse = impl.attention_fwd(q, k, v, causal=False, scale=1.0)
    # row 0: scores 0.5, -1; row 1: scores 1, -2
    e = math.exp
    assert abs(o[0, 0, 0] - (3 * e(0.5) + 5 * e(-1)) / (e(0.5) + e(-1))) < 1e-14
    assert abs(o[1, 0, 0] - (3 * e(1) + 5 * e(-2)) / (e(1) + e(-2))) < 1e-14
    assert abs(lse[0, 0] - math.log(e(0.5) + e(-1))) < 1e-14
    assert abs(lse[0, 1] - math.log(e(1) + e(-2))) < 1e-14
    # causal: row 0 sees only key 0
    o, lse = impl.attention_fwd(q, k, v, causal=True, scale=1.0)
    assert o[0, 0, 0] == 3.0 and lse[0, 0] == 0.5


def check_sampled_rows_match_full():
    T, hq, hkv, d = 50, 4, 2, 8
    cu = [0, 17, 50]
    q, k, v, do = rand_qkv(T, hq, hkv, d, 4)
    o, lse = oracle.attention_fwd(q, k, v, causal=True, cu_seqlens=cu)
    dq, dk, dv, D, _ = oracle.attention_bwd(q, k, v, do, causal=True, cu_seqlens=cu)
    hs, is_ = np.array([0, 3, 1, 2]), np.array([0, 49, 17, 16])
    o_r, l_r = oracle.fwd_rows(q, k, v, hs, is_, causal=True, cu_seqlens=cu)
    assert np.max(np.abs(o_r - o[is_, hs])) == 0.0
    assert np.max(np.abs(l_r - lse[hs, is_])) == 0.0
    gs, js = np.array([1, 0]), np.array([49, 3])
    dk_r, dv_r = oracle.bwd_keys(q, k, v, do, gs, js, causal=True, cu_seqlens=cu)
    assert np.max(np.abs(dk_r - dk[js, gs])) < 1e-14
    assert np.max(np.abs(dv_r - dv[js, gs])) < 1e-14


PINS = {
    "bruteforce": check_bruteforce,
    "fd_gradients": check_fd_gradients,
    "partition_merge": check_partition_merge,
    "merge_rule": check_merge_rule,
    "backward_identities": check_backward_identities,
    "closed_forms": check_closed_forms,
    "dominant_key": check_dominant_key,
    "hand_case": check_hand_case,
    "sampled_rows": check_sampled_rows_match_full,
}


@pytest.mark.parametrize("name", list(PINS))
def test_pin(name):
    PINS[name]()


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_bruteforce_more_seeds(seed):
    check_bruteforce(seed)


def test_mask_matrix_definition():
    """The brute force's mask is block-diagonal lower-triangular for causal
    varlen, block-diagonal for non-causal varlen."""
    cu = [0, 3, 7, 10]
    M = mask_matrix(10, cu, True)
    doc = np.repeat(np.arange(3), np.diff(cu))
    for i in range(10):
        for j in range(10):
            assert M[i, j] == (doc[i] == doc[j] and j <= i)
    assert np.array_equal(mask_matrix(10, None, False), np.ones((10, 10), bool))
