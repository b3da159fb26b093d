"""Seeded synthetic inputs for ring attention, shared by the tests, the bench
and the oracle's callers.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic, so the CUDA path and the fp64 oracle can both be fed
from it without sharing any of the method.

Recipe (the same for every workload):
  * one ``torch.Generator('cpu')`` seeded with ``seed`` draws q, k, v and then
    (when asked) dO, in that order, as fp32 standard normals;
  * each tensor is then cast to the workload's dtype (bf16 rounds to nearest
    even), so the oracle reads exactly the values the GPU reads;
  * problems too large to draw on the host (billions of values) are drawn the
    same way by a generator on the device (``make_qkv_device``): the same
    distribution and order, other values;
  * packed-document lengths come from a second generator seeded ``seed + 1``:
    integers uniform in [lo, hi] inclusive, drawn one at a time until their sum
    reaches the token total, the last one truncated so the sum is exact.

The named workloads mirror the shapes the pages talk about: Llama-3-8B
attention heads (32 query / 8 key-value heads of dimension 128, axolotl
"Sequence Parallelism" page, "Example") at 8K to 64K tokens, with context
parallel degrees 4 and 8 ("Configuration"), and packed samples whose shards
split documents mid-sample ("Sample Packing with Sequence Parallelism").
"""
from __future__ import annotations

import dataclasses

import torch

CONTIGUOUS = 0
ZIGZAG = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    total_tokens: int
    hq: int
    hkv: int
    head_dim: int
    num_shards: int
    layout: int          # CONTIGUOUS or ZIGZAG
    causal: bool
    dtype: str           # "fp32" or "bf16"
    varlen: bool = False  # packed documents, lengths uniform in [doc_lo, doc_hi]
    doc_lo: int = 512
    doc_hi: int = 8192
    backward: bool = False
    heads_k_stride: int = 1
    kv_exchange: int = 0  # 0: ring (batch_ring), 1: all-gather (varlen_llama3)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_fp32_noncausal_t256", 256, 2, 2, 64, 2, CONTIGUOUS,
                 False, "fp32"),
        Workload("causal_mha_t8192_p4_zigzag", 8192, 8, 8, 128, 4, ZIGZAG,
                 True, "bf16"),
        Workload("causal_gqa_t32768_p8_zigzag", 32768, 32, 8, 128, 8, ZIGZAG,
                 True, "bf16"),
        Workload("varlen_causal_gqa_t65536_p8_contiguous", 65536, 32, 8, 128, 8,
                 CONTIGUOUS, True, "bf16", varlen=True),
        # the same packed workload with the page's default exchange under sample
        # packing (varlen_llama3: K/V gathered, heads_k_stride heads at a time)
        Workload("varlen_causal_gqa_t65536_p8_contiguous_allgather", 65536, 32, 8, 128, 8,
                 CONTIGUOUS, True, "bf16", varlen=True, heads_k_stride=2, kv_exchange=1),
        Workload("causal_gqa_fwdbwd_t65536_p8_zigzag", 65536, 32, 8, 128, 8,
                 ZIGZAG, True, "bf16", backward=True),
    ]
}


def torch_dtype(name: str) -> torch.dtype:
    return {"fp32": torch.float32, "bf16": torch.bfloat16}[name]


def doc_lengths(total: int, lo: int, hi: int, seed: int) -> list[int]:
    """Document lengths uniform in [lo, hi], drawn until they cover ``total``;
    the last is truncated so they sum to ``total`` exactly."""
    g = torch.Generator("cpu").manual_seed(seed)
    out: list[int] = []
    acc = 0
    while acc < total:
        n = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
        n = min(n, total - acc)
        out.append(n)
        acc += n
    return out


def cu_seqlens_from_lengths(lengths) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def make_qkv(total_tokens: int, hq: int, hkv: int, head_dim: int, dtype: str,
             seed: int, with_dout: bool = False):
    """q [T,Hq,D], k [T,Hkv,D], v [T,Hkv,D] (and dO [T,Hq,D]) on the CPU."""
    g = torch.Generator("cpu").manual_seed(seed)
    dt = torch_dtype(dtype)
    q = torch.randn(total_tokens, hq, head_dim, generator=g).to(dt)
    k = torch.randn(total_tokens, hkv, head_dim, generator=g).to(dt)
    v = torch.randn(total_tokens, hkv, head_dim, generator=g).to(dt)
    if not with_dout:
        return q, k, v
    do = torch.randn(total_tokens, hq, head_dim, generator=g).to(dt)
    return q, k, v, do


def make_qkv_device(total_tokens: int, hq: int, hkv: int, head_dim: int, seed: int,
                    device, with_dout: bool = False):
    """bf16 q, k, v (and dO) drawn on `device` by a generator seeded `seed`:
    fp32 standard normals in the order q, k, v, dO, each rounded to bf16."""
    g = torch.Generator(device).manual_seed(seed)
    shapes = [(total_tokens, hq, head_dim), (total_tokens, hkv, head_dim),
              (total_tokens, hkv, head_dim)] + ([(total_tokens, hq, head_dim)] if with_dout else [])
    out = []
    for shp in shapes:
        t = torch.empty(shp, dtype=torch.bfloat16, device=device)
        for r0 in range(0, shp[0], 65536):  # fp32 draws a slab at a time
            r1 = min(shp[0], r0 + 65536)
            t[r0:r1] = torch.randn((r1 - r0,) + shp[1:], generator=g, device=device)
        out.append(t)
    return tuple(out)


def make_inputs(w: Workload, seed: int = 0, with_dout: bool | None = None):
    """All inputs of a workload: dict with q, k, v, (dout), cu_seqlens (or None)."""
    wd = w.backward if with_dout is None else with_dout
    t = make_qkv(w.total_tokens, w.hq, w.hkv, w.head_dim, w.dtype, seed, wd)
    out = {"q": t[0], "k": t[1], "v": t[2], "dout": t[3] if wd else None,
           "cu_seqlens": None}
    if w.varlen:
        out["cu_seqlens"] = cu_seqlens_from_lengths(
            doc_lengths(w.total_tokens, w.doc_lo, w.doc_hi, seed + 1))
    return out



# ------------------------------------------------- Mamba2 selective scan
#
# Hybrid models (Nemotron-H, Falcon-H1, Granite; axolotl page, "Mamba/SSM
# Hybrid Models") put Mamba2 layers next to attention.  The synthetic inputs
# follow a Mamba2 layer's usual parameter ranges: dt log-uniform in
# [0.001, 0.1] (the range dt_bias is initialised for), A = -a with a uniform
# in [1, 16] (A_log initialised as log of that range), D = 1, x, B, C standard
# normal; packed samples have the attention workloads' length recipe and
# positions that restart at 0 in each sample.

@dataclasses.dataclass(frozen=True)
class SsdWorkload:
    name: str
    total_tokens: int
    heads: int
    head_dim: int
    state_dim: int
    groups: int
    num_shards: int
    packed: bool = True
    doc_lo: int = 512
    doc_hi: int = 8192


SSD_WORKLOADS = {
    w.name: w for w in [
        # d_inner 8192 (d_model 4096, expand 2) in heads of 64, state 128, 8 groups
        SsdWorkload("mamba2_ssd_t32768_h128_n128_p8", 32768, 128, 64, 128, 8, 8),
    ]
}


def position_ids_from_lengths(lengths) -> torch.Tensor:
    return torch.cat([torch.arange(int(n), dtype=torch.int32) for n in lengths])


def make_ssd_inputs_device(T, H, P, N, G, seed, device, doc_lo=512, doc_hi=8192):
    """make_ssd_inputs' recipe (packed samples) drawn by a generator on
    `device`, for problems too large to draw on the host: the same
    distributions and order, other values; the sample lengths are the host's."""
    g = torch.Generator(device).manual_seed(seed)
    x = torch.randn(T, H, P, generator=g, device=device)
    lo, hi = torch.log(torch.tensor(1e-3)), torch.log(torch.tensor(1e-1))
    dt = torch.exp(lo + (hi - lo) * torch.rand(T, H, generator=g, device=device))
    A = -(1.0 + 15.0 * torch.rand(H, generator=g, device=device))
    B = torch.randn(T, G, N, generator=g, device=device)
    C = torch.randn(T, G, N, generator=g, device=device)
    D = torch.ones(H, device=device)
    pos = position_ids_from_lengths(doc_lengths(T, doc_lo, doc_hi, seed + 1)).to(device)
    return {"x": x, "dt": dt, "A": A, "B": B, "C": C, "D": D, "position_ids": pos}


def make_ssd_inputs(T, H, P, N, G, seed, packed=True, doc_lo=512, doc_hi=8192):
    """x [T,H,P], dt [T,H], A [H], B, C [T,G,N], D [H] (fp32, CPU) and
    position_ids [T] int32 (None when not packed)."""
    g = torch.Generator("cpu").manual_seed(seed)
    x = torch.randn(T, H, P, generator=g)
    lo, hi = torch.log(torch.tensor(1e-3)), torch.log(torch.tensor(1e-1))
    dt = torch.exp(lo + (hi - lo) * torch.rand(T, H, generator=g))
    A = -(1.0 + 15.0 * torch.rand(H, generator=g))
    B = torch.randn(T, G, N, generator=g)
    C = torch.randn(T, G, N, generator=g)
    D = torch.ones(H)
    pos = None
    if packed:
        pos = position_ids_from_lengths(doc_lengths(T, doc_lo, doc_hi, seed + 1))
    return {"x": x, "dt": dt, "A": A, "B": B, "C": C, "D": D, "position_ids": pos}
