"""GPU parity of the context-parallel Mamba2 selective scan against the fp64
oracle's scan over the whole, unsharded sequence.

Every case runs through the C ABI (ssd_cp_fwd): the chunks of num_shards
virtual ranks are scanned from a zero state, the final states are passed
along the ring and the additive correction is applied (axolotl page,
"Mamba/SSM Hybrid Models").  Outputs are pre-filled with NaN.
"""
import numpy as np
import pytest
import torch

import context_long_sequence_fwd_b300 as ra
import oracle
from context_long_sequence_fwd_b300.workloads import (SSD_WORKLOADS, make_ssd_inputs,
                                                      make_ssd_inputs_device,
                                                      position_ids_from_lengths)
from tests._util import max_err, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
# fp32-level arithmetic against fp64 (state size 64: fp32 on CUDA cores;
# state size 128: fp16 hi + lo split products, three per term, about 2^-22
# of each product, accumulated in fp32): each output sums at most a few
# hundred decayed terms of magnitude ~1 (dt <= 0.1, |A| >= 1), so the
# rounding stays below 1e-5 relative to the outputs' scale.
REL_TOL = 2e-5


def run(inp, R, want_state=True):
    t = {k: (None if v is None else v.to(DEV)) for k, v in inp.items()}
    y = torch.full(t["x"].shape, float("nan"), device=DEV)
    y, hT = ra.ssd_cp_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["position_ids"], R,
                          y=y, want_final_state=want_state)
    assert ra.ringattn_get_status() == 0
    return to_np(y), None if hT is None else to_np(hT)


def check(inp, R):
    y, hT = run(inp, R)
    ry, rh = oracle.ssd_scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                             inp["position_ids"])
    scale = max(1.0, float(np.max(np.abs(ry))))
    assert max_err(y, ry) <= REL_TOL * scale, (max_err(y, ry), scale)
    hs = max(1.0, float(np.max(np.abs(rh))))
    assert max_err(hT, rh) <= REL_TOL * hs, (max_err(hT, rh), hs)


CASES = [
    # T, H, N, G, R, packed lengths (None: one sample)
    (256, 2, 64, 1, 1, None),
    (256, 4, 64, 2, 2, None),
    (1000, 4, 128, 2, 4, None),                  # chunks of 250: ragged token blocks
    (2048, 4, 128, 4, 8, [300, 5, 1, 700, 1042]),
    (2048, 8, 64, 2, 8, [100] * 20 + [48]),       # samples shorter than a chunk
    (1536, 2, 128, 1, 3, [1536]),                 # positions from 0, one sample
    (384, 2, 128, 1, 4, None),                    # chunks of 96: shorter than a 128-token block
    (600, 4, 128, 2, 8, [37, 200, 1, 362]),       # chunks of 75 with sample starts inside
    (512, 2, 128, 1, 1, None),                    # one rank: no state passing, no correction
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_scan_matches_oracle(case):
    T, H, N, G, R, lengths = case
    inp = make_ssd_inputs(T, H, 64, N, G, seed=3, packed=False)
    if lengths is not None:
        inp["position_ids"] = position_ids_from_lengths(lengths)
    check(inp, R)


def test_chunk_starting_mid_sample():
    """Positions that do not start at 0: the first sample began before this
    sequence, and its state is taken as zero (nothing before token 0)."""
    T = 1024
    inp = make_ssd_inputs(T, 4, 64, 64, 2, seed=5, packed=False)
    inp["position_ids"] = torch.cat([torch.arange(300, 600, dtype=torch.int32),
                                     torch.arange(724, dtype=torch.int32)])
    check(inp, 4)


def test_without_skip_term():
    inp = make_ssd_inputs(512, 2, 64, 64, 1, seed=6, packed=False)
    inp["D"] = None
    check(inp, 4)


@pytest.mark.parametrize("lo,hi", [(0.3, 1.0), (0.01, 10.0)])
def test_strong_decay(lo, hi):
    """Decays strong enough that a 32-token block's running decay product
    falls below 1e-20: the scan rebases its scaled state (dt A about -5 per
    token), or drops the previous state outright where one token's decay is
    itself below 1e-20 (dt A down to -160)."""
    T, H = 1024, 4
    inp = make_ssd_inputs(T, H, 64, 128, 2, seed=9, packed=False)
    g = torch.Generator("cpu").manual_seed(19)
    inp["dt"] = torch.exp(torch.empty(T, H).uniform_(np.log(lo), np.log(hi), generator=g))
    inp["A"] = -torch.empty(H).uniform_(5.0, 16.0, generator=g)
    check(inp, 4)


def test_shards_do_not_change_the_result():
    inp = make_ssd_inputs(4096, 4, 64, 128, 2, seed=7)
    y1, h1 = run(inp, 1)
    for R in (2, 8, 16):
        yR, hR = run(inp, R)
        scale = max(1.0, float(np.max(np.abs(y1))))
        assert max_err(yR, y1) <= REL_TOL * scale


def test_mamba2_workload_every_head():
    """The full 32K-token, 128-head workload against one oracle scan of every
    head over the whole sequence; each head is checked against its own
    outputs' scale."""
    w = SSD_WORKLOADS["mamba2_ssd_t32768_h128_n128_p8"]
    inp = make_ssd_inputs(w.total_tokens, w.heads, w.head_dim, w.state_dim, w.groups, seed=0)
    y, hT = run(inp, w.num_shards)
    ry, rh = oracle.ssd_scan(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                             inp["position_ids"])
    ry, rh = np.asarray(ry), np.asarray(rh)
    for h in range(w.heads):
        scale = max(1.0, float(np.max(np.abs(ry[:, h]))))
        assert max_err(y[:, h], ry[:, h]) <= REL_TOL * scale, h
        assert max_err(hT[h], rh[h]) <= REL_TOL * max(1.0, float(np.max(np.abs(rh[h])))), h
    assert np.all(np.isfinite(y))


def test_mamba2_t1048576_past_int32_offsets():
    """The 32K workload's shape at 1,048,576 tokens: x and y hold 2^20 x 128 x
    64 = 8.6e9 values each (byte offsets past 2^34), drawn on the device.
    Heads 0 and 127 (groups 0 and 7) are checked in full, every y and the
    final state, against the oracle's scan of each head as its own problem
    (heads are independent given their group's B and C)."""
    T, H, P, N, G, R = 1 << 20, 128, 64, 128, 8, 8
    inp = make_ssd_inputs_device(T, H, P, N, G, seed=4, device=DEV)
    y, hT = ra.ssd_cp_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                          inp["position_ids"], R, want_final_state=True)
    torch.cuda.synchronize()
    assert ra.ringattn_get_status() == 0
    pos = inp["position_ids"].cpu()
    for h in (0, H - 1):
        g = h // (H // G)
        sub = lambda t: t.contiguous().cpu().double().numpy()
        ry, rh = oracle.ssd_scan(sub(inp["x"][:, h:h + 1]), sub(inp["dt"][:, h:h + 1]),
                                 sub(inp["A"][h:h + 1]), sub(inp["B"][:, g:g + 1]),
                                 sub(inp["C"][:, g:g + 1]), sub(inp["D"][h:h + 1]), pos)
        ry, rh = np.asarray(ry)[:, 0], np.asarray(rh)[0]
        scale = max(1.0, float(np.max(np.abs(ry))))
        assert max_err(to_np(y[:, h]), ry) <= REL_TOL * scale, h
        assert max_err(to_np(hT[h]), rh) <= REL_TOL * max(1.0, float(np.max(np.abs(rh)))), h
    assert bool(torch.isfinite(y).all())


def test_bad_arguments_are_loud():
    x = torch.zeros(100, 2, 64, device=DEV)
    dt = torch.zeros(100, 2, device=DEV)
    A = torch.zeros(2, device=DEV)
    B = torch.zeros(100, 1, 64, device=DEV)
    with pytest.raises(ra.RingAttnError) as e:
        ra.ssd_cp_fwd(x, dt, A, B, B, num_shards=3)
    assert e.value.code == -2
    B2 = torch.zeros(100, 1, 32, device=DEV)
    with pytest.raises(ra.RingAttnError) as e:
        ra.ssd_cp_fwd(x, dt, A, B2, B2, num_shards=2)
    assert e.value.code == -3
