"""GPU parity of attn_lse_merge (the ring-step aggregation) against the oracle's
merge, and of merging per-shard partials into full attention."""
import numpy as np
import pytest
import torch

import context_long_sequence_fwd_b300 as ra
import oracle
from context_long_sequence_fwd_b300.workloads import make_qkv
from tests._util import TOL_BF16_O, TOL_FP32, max_err, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def partials(rows, heads, d, seed, dtype):
    g = torch.Generator("cpu").manual_seed(seed)
    oa = torch.randn(rows, heads, d, generator=g).to(dtype)
    ob = torch.randn(rows, heads, d, generator=g).to(dtype)
    la = torch.randn(heads, rows, generator=g) * 4
    lb = torch.randn(heads, rows, generator=g) * 4
    # empty sides: one, the other, both (an empty partial has O = 0)
    la[0, 0] = -float("inf")
    lb[0, 1] = -float("inf")
    la[0, 2] = lb[0, 2] = -float("inf")
    oa[0, 0] = 0
    ob[1, 0] = 0
    oa[2, 0] = 0
    ob[2, 0] = 0
    return oa, la, ob, lb


@pytest.mark.parametrize("dtype,tol", [(torch.float32, TOL_FP32), (torch.bfloat16, None)])
@pytest.mark.parametrize("rows,heads,d", [(1000, 3, 128), (37, 2, 64), (4096, 8, 128), (300, 3, 8),
                                          (129, 2, 16), (77, 5, 32), (64, 2, 256)])
def test_merge_matches_oracle(dtype, tol, rows, heads, d):
    oa, la, ob, lb = partials(rows, heads, d, 7, dtype)
    ro, rl = oracle.lse_merge(oa.permute(1, 0, 2), la, ob.permute(1, 0, 2), lb)
    a_o, a_l = oa.to(DEV), la.to(DEV)
    ra.attn_lse_merge(a_o, a_l, ob.to(DEV), lb.to(DEV))
    assert ra.ringattn_get_status() == 0
    go = to_np(a_o).transpose(1, 0, 2)
    gl = to_np(a_l)
    assert max_err(gl, rl) <= 1e-5
    if tol is not None:
        assert max_err(go, ro) <= tol
    else:
        # bf16 output: rounding to nearest costs at most half an ulp, 2^-8 |x|
        fin = np.isfinite(ro)
        assert np.all(np.abs(go - ro)[fin] <= np.abs(ro[fin]) * 2.0 ** -8 * 1.01 + 1e-5)
    assert np.all(go[0, 2] == 0) and gl[0, 2] == -np.inf


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_merge_empty_side_is_ignored_exactly(dtype):
    """A side with lse = -inf contributes nothing, whatever its o holds (here
    NaN and inf): the other side comes through bit for bit."""
    rows, heads, d = 513, 4, 128
    oa, la, ob, lb = partials(rows, heads, d, 3, dtype)
    la[:, :] = torch.randn(heads, rows)
    lb[:, :] = -float("inf")
    lb[:, ::3] = torch.randn(heads, (rows + 2) // 3)
    la[:, ::3] = -float("inf")
    ob[1::3] = float("nan")
    ob[2::3] = float("inf")
    oa[0::3] = float("nan")
    a_o, a_l = oa.to(DEV), la.to(DEV)
    ra.attn_lse_merge(a_o, a_l, ob.to(DEV), lb.to(DEV))
    assert ra.ringattn_get_status() == 0
    go, gl = a_o.cpu(), a_l.cpu()
    keep_b = torch.zeros(rows, dtype=torch.bool)
    keep_b[::3] = True
    assert torch.equal(go[keep_b], ob[keep_b]) and torch.equal(go[~keep_b], oa[~keep_b])
    assert torch.equal(gl[:, keep_b], lb[:, keep_b]) and torch.equal(gl[:, ~keep_b], la[:, ~keep_b])


def test_merge_of_shard_partials_is_attention():
    """Per-shard partial attention (oracle, fp64 -> fp32) merged on the GPU in
    ring order equals attention over the whole sequence."""
    T, hq, hkv, d, P = 512, 4, 2, 64, 4
    q, k, v = make_qkv(T, hq, hkv, d, "fp32", seed=1)
    full_o, full_l = oracle.attention_fwd(q, k, v, causal=True)
    C = T // P
    acc_o = acc_l = None
    for s in range(P):
        allowed = (np.arange(T) // C) == (P - 1 - s)
        po, pl = oracle.attention_fwd(q, k, v, causal=True, key_allowed=allowed)
        po_t = torch.tensor(po, dtype=torch.float32, device=DEV)
        pl_t = torch.tensor(pl, dtype=torch.float32, device=DEV)
        if acc_o is None:
            acc_o, acc_l = po_t, pl_t
        else:
            ra.attn_lse_merge(acc_o, acc_l, po_t, pl_t)
    assert max_err(to_np(acc_o), full_o) <= TOL_FP32
    assert max_err(to_np(acc_l), full_l) <= TOL_FP32


def test_merge_rejects_bad_args():
    x = torch.zeros(8, 2, 12, device=DEV)
    l = torch.zeros(2, 8, device=DEV)
    with pytest.raises(ra.RingAttnError):
        ra.attn_lse_merge(x, l, x.clone(), l.clone())
