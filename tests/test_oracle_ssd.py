"""Pins for the fp64 SSD (Mamba2 selective scan) oracle, checked against
things other than its own recurrence.

* brute force on tiny inputs: the scan's closed form as a sum over past
  tokens -- y_t = sum_{s <= t, same sample} (C_t . B_s) dt_s
  exp(A sum_{s < u <= t} dt_u) x_s + D x_t, plus the initial state's decayed
  contribution while no sample boundary intervenes -- built with numpy;
* closed forms: one token; a decay so strong that only the current token
  counts;
* the context-parallel identity the GPU path relies on (the axolotl page,
  "Mamba/SSM Hybrid Models": each rank scans its chunk, passes its final
  state on, and an additive correction accounts for the state it did not
  start from): scanning a prefix and continuing from its final state equals
  scanning the whole sequence, and a scan from h0 equals the scan from zero
  plus the decayed h0 read out through C;
* packed samples: outputs of a sample do not depend on an earlier sample.
"""
import math

import numpy as np
import pytest

import oracle


def rand_ssd(T, H, P, N, G, seed, with_D=True):
    r = np.random.default_rng(seed)
    x = r.standard_normal((T, H, P))
    dt = np.log1p(np.exp(r.standard_normal((T, H))))  # softplus: positive
    A = -np.exp(r.standard_normal(H) * 0.5)            # negative decay rates
    B = r.standard_normal((T, G, N))
    C = r.standard_normal((T, G, N))
    D = r.standard_normal(H) if with_D else None
    return x, dt, A, B, C, D


def sample_starts(T, pos):
    """Start token of the sample holding each token (pos == 0 starts one)."""
    st = np.zeros(T, np.int64)
    cur = 0
    for t in range(T):
        if pos is not None and pos[t] == 0:
            cur = t
        st[t] = cur
    return st


def brute_force(x, dt, A, B, C, D, pos=None, h0=None):
    T, H, P = x.shape
    G = B.shape[1]
    st = sample_starts(T, pos)
    y = np.zeros_like(x)
    cum = np.concatenate([np.zeros((1, H)), np.cumsum(dt, 0)])  # cum[t] = sum_{u < t} dt_u
    for h in range(H):
        g = h // (H // G)
        for t in range(T):
            acc = np.zeros(P)
            for s in range(st[t], t + 1):
                decay = math.exp(A[h] * (cum[t + 1, h] - cum[s + 1, h]))
                acc += float(C[t, g] @ B[s, g]) * dt[s, h] * decay * x[s, h]
            if h0 is not None and st[t] == 0 and (pos is None or pos[0] != 0):
                acc += math.exp(A[h] * cum[t + 1, h]) * (h0[h] @ C[t, g])
            y[t, h] = acc + (0.0 if D is None else D[h]) * x[t, h]
    return y


CASES = [
    # T, H, P, N, G, pos
    (12, 2, 3, 4, 1, None),
    (20, 4, 5, 3, 2, None),
    (24, 2, 4, 6, 2, [0, 1, 2, 3, 4, 0, 1, 2, 0, 1, 2, 3, 4, 5, 6, 7, 0, 1, 2, 3, 4, 5, 6, 7]),
    (16, 3, 2, 5, 3, [3, 4, 5, 0, 1, 2, 3, 0, 0, 1, 2, 3, 4, 5, 6, 7]),  # starts mid-sample
]


def check_bruteforce(seed=0):
    for T, H, P, N, G, pos in CASES:
        x, dt, A, B, C, D = rand_ssd(T, H, P, N, G, seed)
        y, _ = oracle.ssd_scan(x, dt, A, B, C, D, pos)
        assert np.max(np.abs(y - brute_force(x, dt, A, B, C, D, pos))) < 1e-11
        h0 = np.random.default_rng(seed + 7).standard_normal((H, P, N))
        y, _ = oracle.ssd_scan(x, dt, A, B, C, D, pos, h0=h0)
        assert np.max(np.abs(y - brute_force(x, dt, A, B, C, D, pos, h0))) < 1e-11


def check_closed_forms():
    x, dt, A, B, C, D = rand_ssd(1, 2, 3, 4, 1, 3)
    y, hT = oracle.ssd_scan(x, dt, A, B, C, D)
    for h in range(2):
        want = dt[0, h] * float(B[0, 0] @ C[0, 0]) * x[0, h] + D[h] * x[0, h]
        assert np.max(np.abs(y[0, h] - want)) < 1e-14
        assert np.max(np.abs(hT[h] - dt[0, h] * np.outer(x[0, h], B[0, 0]))) < 1e-14
    # decay so strong that every earlier token is forgotten
    x, dt, A, B, C, D = rand_ssd(10, 2, 3, 4, 1, 4)
    A = np.full(2, -1e4)
    dt = dt + 0.5
    y, _ = oracle.ssd_scan(x, dt, A, B, C, D)
    for t in range(10):
        for h in range(2):
            want = dt[t, h] * float(B[t, 0] @ C[t, 0]) * x[t, h] + D[h] * x[t, h]
            assert np.max(np.abs(y[t, h] - want)) < 1e-12


def check_state_passing():
    T, H, P, N, G = 40, 2, 4, 5, 1
    x, dt, A, B, C, D = rand_ssd(T, H, P, N, G, 5)
    pos = list(range(13)) + list(range(27))      # a sample starts at token 13
    y, hT = oracle.ssd_scan(x, dt, A, B, C, D, pos)
    for cut in (7, 13, 20, 33):
        ya, ha = oracle.ssd_scan(x[:cut], dt[:cut], A, B[:cut], C[:cut], D, pos[:cut])
        yb, hb = oracle.ssd_scan(x[cut:], dt[cut:], A, B[cut:], C[cut:], D, pos[cut:], h0=ha)
        assert np.max(np.abs(np.concatenate([ya, yb]) - y)) < 1e-12
        assert np.max(np.abs(hb - hT)) < 1e-12
        # linearity in the initial state: zero-start scan + decayed h0 through C
        y0, _ = oracle.ssd_scan(x[cut:], dt[cut:], A, B[cut:], C[cut:], D, pos[cut:])
        first_reset = next((i for i, p in enumerate(pos[cut:]) if p == 0), T - cut)
        corr = np.zeros_like(y0)
        for h in range(H):
            lam = np.cumsum(dt[cut:, h]) * A[h]
            for i in range(first_reset):
                corr[i, h] = math.exp(lam[i]) * (ha[h] @ C[cut + i, 0])
        assert np.max(np.abs(y0 + corr - yb)) < 1e-12


def check_samples_independent():
    T, H, P, N, G = 30, 2, 3, 4, 1
    x, dt, A, B, C, D = rand_ssd(T, H, P, N, G, 6)
    pos = list(range(11)) + list(range(19))
    y, _ = oracle.ssd_scan(x, dt, A, B, C, D, pos)
    x2 = x.copy()
    x2[:11] += 5.0
    B2 = B.copy()
    B2[:11] *= -2.0
    y2, _ = oracle.ssd_scan(x2, dt, A, B2, C, D, pos)
    assert np.max(np.abs(y2[11:] - y[11:])) == 0.0
    assert np.max(np.abs(y2[:11] - y[:11])) > 1e-3


PINS = {
    "bruteforce": check_bruteforce,
    "closed_forms": check_closed_forms,
    "state_passing": check_state_passing,
    "samples_independent": check_samples_independent,
}


@pytest.mark.parametrize("name", list(PINS))
def test_pin(name):
    PINS[name]()


@pytest.mark.parametrize("seed", [1, 2])
def test_bruteforce_more_seeds(seed):
    check_bruteforce(seed)
