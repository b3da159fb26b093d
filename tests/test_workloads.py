"""The seeded input generators (no attention or scan arithmetic in them):
shapes, dtypes, distributions and determinism of the host and device draws.
The device draws run here on the CPU device; on a GPU they run the same
code with a CUDA generator."""
import torch

from context_long_sequence_fwd_b300.workloads import (doc_lengths, make_qkv, make_qkv_device,
                                                      make_ssd_inputs_device)


def test_host_draws_are_seeded_and_rounded_to_bf16():
    a = make_qkv(512, 4, 2, 64, "bf16", seed=7, with_dout=True)
    b = make_qkv(512, 4, 2, 64, "bf16", seed=7, with_dout=True)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert [tuple(t.shape) for t in a] == [(512, 4, 64), (512, 2, 64), (512, 2, 64), (512, 4, 64)]
    assert all(t.dtype == torch.bfloat16 for t in a)


def test_device_draws_follow_the_same_recipe():
    """q, k, v, dO drawn in slabs of 65536 rows: standard normals rounded to
    bf16, the same for the same seed, different for another."""
    a = make_qkv_device(70000, 2, 1, 64, seed=1, device="cpu", with_dout=True)
    b = make_qkv_device(70000, 2, 1, 64, seed=1, device="cpu", with_dout=True)
    c = make_qkv_device(70000, 2, 1, 64, seed=2, device="cpu")
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert not torch.equal(a[0], c[0])
    assert [tuple(t.shape) for t in a] == [(70000, 2, 64), (70000, 1, 64), (70000, 1, 64),
                                           (70000, 2, 64)]
    for t in a:
        assert t.dtype == torch.bfloat16
        f = t.float()
        assert abs(float(f.mean())) < 0.02 and abs(float(f.std()) - 1.0) < 0.02


def test_device_ssd_draws_follow_the_recipe():
    d = make_ssd_inputs_device(20000, 4, 64, 128, 2, seed=3, device="cpu")
    assert tuple(d["x"].shape) == (20000, 4, 64) and tuple(d["B"].shape) == (20000, 2, 128)
    assert float(d["dt"].min()) >= 1e-3 * (1 - 1e-6) and float(d["dt"].max()) <= 1e-1 * (1 + 1e-6)
    assert float(d["A"].max()) <= -1.0 and float(d["A"].min()) >= -16.0
    assert torch.equal(d["D"], torch.ones(4))
    # positions restart at 0 at each packed sample, whose lengths are the host's draw
    pos = d["position_ids"]
    starts = (pos == 0).nonzero().flatten().tolist()
    lengths = [b - a for a, b in zip(starts, starts[1:] + [20000])]
    assert lengths == doc_lengths(20000, 512, 8192, 4)
