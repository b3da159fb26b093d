"""Pins for the matrix-product oracle (``oracle.blas``).

The fp64 oracle that uses library matrix products is pinned like the C
oracle, by things other than itself:

* every definition-level pin of test_oracle.py (brute force with an explicit
  mask matrix and scipy's softmax, finite differences of the gradients, the
  partition-merge identity of ring steps, D = dO . O and the sums of dK and
  dV, the closed forms, a dominant key, the hand-worked D = 1 case) runs on it;
* it agrees with the independently written C oracle to rounding on random
  problems with GQA, packed documents (empty ones included) and both masks;
* planted mistakes in a copy of its source are each caught by a pin.
"""
import importlib.util
import os

import numpy as np
import pytest

import oracle
from tests import test_oracle as pins

BLAS_PINS = {
    "bruteforce": pins.check_bruteforce,
    "fd_gradients": pins.check_fd_gradients,
    "partition_merge": pins.check_partition_merge,
    "backward_identities": pins.check_backward_identities,
    "closed_forms": pins.check_closed_forms,
    "dominant_key": pins.check_dominant_key,
    "hand_case": pins.check_hand_case,
}


@pytest.mark.parametrize("name", list(BLAS_PINS))
def test_pin(name):
    BLAS_PINS[name](impl=oracle.blas)


@pytest.mark.parametrize("seed", [1, 2])
def test_bruteforce_more_seeds(seed):
    pins.check_bruteforce(seed, impl=oracle.blas)


AGREE_CASES = [
    # T, hq, hkv, d, cu_seqlens, causal
    (300, 4, 2, 16, None, True),
    (257, 6, 2, 8, [0, 10, 11, 100, 257], True),
    (200, 3, 1, 8, [0, 50, 200], False),
    (96, 2, 1, 4, [0, 0, 30, 30, 96], True),
    (130, 8, 1, 8, [0, 1, 2, 3, 130], True),
]


@pytest.mark.parametrize("case", AGREE_CASES, ids=str)
def test_agrees_with_c_oracle(case):
    T, hq, hkv, d, cu, causal = case
    q, k, v, do = pins.rand_qkv(T, hq, hkv, d, 17)
    o1, l1 = oracle.attention_fwd(q, k, v, causal=causal, cu_seqlens=cu)
    o2, l2 = oracle.blas.attention_fwd(q, k, v, causal=causal, cu_seqlens=cu)
    assert np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12
    ref = oracle.attention_bwd(q, k, v, do, causal=causal, cu_seqlens=cu)
    got = oracle.blas.attention_bwd(q, k, v, do, causal=causal, cu_seqlens=cu, return_out=True)
    for a, b in zip(ref, got[:5]):
        assert np.max(np.abs(a - b)) < 1e-12
    assert np.max(np.abs(got[5] - o1)) < 1e-12


def test_head_subsets_leave_the_rest_nan():
    T, hq, hkv, d = 64, 6, 3, 8
    q, k, v, do = pins.rand_qkv(T, hq, hkv, d, 3)
    o, l = oracle.blas.attention_fwd(q, k, v, causal=True, heads=[1, 4])
    full_o, full_l = oracle.blas.attention_fwd(q, k, v, causal=True)
    assert np.array_equal(o[:, [1, 4]], full_o[:, [1, 4]])
    assert np.isnan(o[:, [0, 2, 3, 5]]).all() and np.isnan(l[[0, 2, 3, 5]]).all()
    dq, dk, dv, D, lse = oracle.blas.attention_bwd(q, k, v, do, causal=True, kv_heads=[2])
    ref = oracle.blas.attention_bwd(q, k, v, do, causal=True)
    assert np.array_equal(dk[:, 2], ref[1][:, 2]) and np.array_equal(dq[:, 4:], ref[0][:, 4:])
    assert np.isnan(dk[:, :2]).all() and np.isnan(dq[:, :4]).all()


# ----------------------------------------------------------- planted mistakes

SRC = os.path.join(os.path.dirname(oracle.__file__), "attention_blas.py")

MUTANTS = {
    "causal_excludes_diagonal": ("vis &= j <= i", "vis &= j < i"),
    "lse_drops_max": ("m + torch.log(z)", "torch.log(z)"),
    "fwd_no_scale": ("S = (Qh[rows] @ KgT[:, keys]).mul_(sc)\n            vis = _mask(doc, rows, keys, causal, ka)",
                     "S = (Qh[rows] @ KgT[:, keys])\n            vis = _mask(doc, rows, keys, causal, ka)"),
    "fwd_gqa_wrong_head": ("        g = h // G\n        Qh", "        g = h % hkv\n        Qh"),
    "doc_compare": ("doc[rows][:, None] == doc[keys][None, :]",
                    "doc[rows][:, None] >= doc[keys][None, :]"),
    "weights_not_normalised": (
        "P = E.div_(torch.where(empty, torch.ones_like(z), z)[:, None])", "P = E"),
    "causal_span_drops_last_key": ("k1 = r1 if causal else", "k1 = r1 - 1 if causal else"),
    "dS_wrong_sign": ("dS = dP.sub_(Dr[:, None]).mul_(P)", "dS = dP.add_(Dr[:, None]).mul_(P)"),
    "D_without_P": ("Dr = (P * dP).sum(dim=1)", "Dr = dP.sum(dim=1)"),
    "dq_no_scale": ("(dS @ Kg[keys]).mul_(sc)", "(dS @ Kg[keys])"),
    "dv_wrong_operand": ("acc_v += P.T @ dOs[h][rows]", "acc_v += P.T @ Qs[h][rows]"),
    "dk_drops_D": ("dS = dP.sub_(Ds[h][rows][:, None]).mul_(P)", "dS = dP.mul_(P)"),
    "key_side_skips_first_row": ("i0 = j0 if causal else", "i0 = j0 + 1 if causal else"),
    "dk_no_scale": ("acc_k.mul_(sc).numpy()", "acc_k.numpy()"),
}


def load_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"blas_{name}.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"blas_mutant_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    mod = load_mutant(tmp_path, name)
    failed = []
    for pin_name, fn in BLAS_PINS.items():
        try:
            fn(impl=mod)
        except AssertionError:
            failed.append(pin_name)
    assert failed, f"no pin caught mutant {name}"
