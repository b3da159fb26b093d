"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch

# Acceptance bounds for the ring-attention outputs (max absolute error
# against the fp64 oracle): bf16 operands with fp32 accumulation, and the
# fp32 path.
TOL_BF16_O = 2e-2
TOL_BF16_LSE = 1e-3
TOL_FP32 = 1e-5


def to_np(t):
    t = t.detach().to("cpu")
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.numpy().astype(np.float64)


def max_err(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):  # inf - inf where both_inf masks it out
        d = np.where(both_inf, 0.0, np.abs(a - b))
    return float(np.max(d)) if d.size else 0.0


def nan_like(t):
    out = torch.empty_like(t)
    out.fill_(float("nan"))
    return out


def sample_rows(T, hq, n, seed, extra_rows=()):
    """n random (head, row) pairs plus every head at the given rows."""
    r = np.random.default_rng(seed)
    hs = list(r.integers(0, hq, n))
    is_ = list(r.integers(0, T, n))
    for i in extra_rows:
        for h in range(hq):
            hs.append(h)
            is_.append(int(i))
    return np.array(hs, np.int32), np.array(is_, np.int32)
