"""The C-ABI library loads without a GPU and exports every function that
include/ringattn.h declares; argument errors come back synchronously."""
import ctypes
import os
import re

import numpy as np
import pytest

import context_long_sequence_fwd_b300 as ra
from context_long_sequence_fwd_b300 import build as ra_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ra.LIB_PATH):
        ra_build.build()
    return ra.library()


def declared_functions():
    names = set()
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if not hdr.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("ringattn_fwd", "ringattn_bwd", "attn_lse_merge", "ringattn_fwd_stepwise",
              "ringattn_get_status", "ringattn_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    assert lib.ringattn_status_string(0) == b"ok"
    assert b"divisible" in lib.ringattn_status_string(-2)
    assert lib.ringattn_version() >= 100


def dims(T=256, hq=2, hkv=2, d=128, dtype=ra.RA_BF16, hks=1, nseq=0):
    return ra.ra_dims(T, nseq, hq, hkv, d, dtype, hks, 0)


def test_argument_errors_without_gpu(lib):
    f = lib.ringattn_fwd
    # sizes that do not split into equal chunks
    assert f(None, None, None, None, dims(T=250), 4, ra.CONTIGUOUS, 1, None, None, None) == -2
    assert f(None, None, None, None, dims(T=256), 3, ra.ZIGZAG, 1, None, None, None) == -2
    # heads, dtype, head_dim
    assert f(None, None, None, None, dims(hq=3, hkv=2), 1, 0, 1, None, None, None) == -1
    assert f(None, None, None, None, dims(d=96), 1, 0, 1, None, None, None) == -3
    assert f(None, None, None, None, dims(d=256), 1, 0, 1, None, None, None) == -3
    # bf16 at head_dim 64 is supported: with null tensors it fails as a null argument
    assert f(None, None, None, None, dims(d=64), 1, 0, 1, None, None, None) == -1
    assert f(None, None, None, None, dims(dtype=7), 1, 0, 1, None, None, None) == -3
    assert f(None, None, None, None, dims(hks=3, hkv=2), 1, 0, 1, None, None, None) == -1
    # null tensors with a non-empty problem
    assert f(None, None, None, None, dims(), 1, 0, 1, None, None, None) == -1
    # empty problem: nothing to do
    assert f(None, None, None, None, dims(T=0), 2, ra.ZIGZAG, 1, None, None, None) == 0
    # bad cu_seqlens (must run 0 .. T without decreasing)
    cu = np.array([0, 100, 50, 256], np.int32)
    p = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    assert f(None, None, None, p, dims(nseq=3), 1, 0, 1, None, None, None) == -1
    # workspace checks come before any device work
    assert lib.ringattn_fwd_stepwise(16, 16, 16, None, dims(), 1, 0, 1, 16, 16, None, 0, None) == -6
    assert lib.attn_lse_merge(None, None, None, None, 4, 2, 12, 0, None) == -1
    assert lib.attn_lse_merge(None, None, None, None, 0, 2, 64, 0, None) == 0


def test_ssd_argument_errors_without_gpu(lib):
    f = lib.ssd_cp_fwd
    sd = ra.ssd_dims(1024, 4, 64, 128, 2)
    ws = lib.ssd_cp_workspace_size(sd, 4)
    # (fake) device pointers: every check below comes before any device work
    ok = [256, 512, 768, 1024, 1280, None, None]
    assert f(*ok, ra.ssd_dims(1000, 4, 64, 128, 2), 3, 1536, None, None, ws, None) == -2
    assert f(*ok, ra.ssd_dims(1024, 4, 64, 96, 2), 4, 1536, None, None, ws, None) == -3
    assert f(*ok, ra.ssd_dims(1024, 3, 64, 128, 2), 4, 1536, None, None, ws, None) == -1
    assert f(*ok, sd, 4, 1536, None, None, 0, None) == -6          # no workspace
    # x, B, C and y are moved in 16-byte pieces
    for i in (0, 3, 4):
        bad = list(ok)
        bad[i] += 4
        assert f(*bad, sd, 4, 1536, None, None, ws, None) == -1
    assert f(*ok, sd, 4, 1540, None, None, ws, None) == -1
    assert f(*ok, ra.ssd_dims(0, 4, 64, 128, 2), 4, 1536, None, None, ws, None) == 0


def test_workspace_sizes(lib):
    d = dims(T=1024, hq=4, hkv=2)
    assert lib.ringattn_fwd_stepwise_workspace_size(d) >= 2 * (1024 * 4 * 128 * 4 + 4 * 1024 * 4)
    assert lib.ringattn_bwd_workspace_size(d) >= 4 * 1024 * 4   # the D_i vector


def test_bwd_flush_interval_sizes_the_workspace(lib):
    """bf16 gradients whose key-tile walks (T / 128 query tiles x G heads)
    outlast the dK/dV flush interval need fp32 sums of dk and dv in the
    workspace; fp32 gradients take the flushes themselves."""
    d_vec = lambda T, hq: (hq * T * 4 + 255) // 256 * 256
    sums = lambda T, hkv: 2 * ((T * hkv * 128 * 4 + 255) // 256 * 256)
    try:
        assert lib.ringattn_set_bwd_flush_interval(-1) == -1
        assert lib.ringattn_set_bwd_flush_interval(1024) == 0
        # 256 query tiles x 4 heads = 1024 pairs: no flush at 32K tokens
        assert lib.ringattn_bwd_workspace_size(dims(T=32768, hq=32, hkv=8)) == d_vec(32768, 32)
        big = dims(T=65536, hq=32, hkv=8)
        assert lib.ringattn_bwd_workspace_size(big) == d_vec(65536, 32) + sums(65536, 8)
        big.grad_fp32 = 1
        assert lib.ringattn_bwd_workspace_size(big) == d_vec(65536, 32)
        assert lib.ringattn_set_bwd_flush_interval(0) == 0  # off
        assert lib.ringattn_bwd_workspace_size(dims(T=65536, hq=32, hkv=8)) == d_vec(65536, 32)
        assert lib.ringattn_set_bwd_flush_interval(4) == 0
        assert lib.ringattn_bwd_workspace_size(dims(T=1024, hq=4, hkv=2)) == \
            d_vec(1024, 4) + sums(1024, 2)
    finally:
        lib.ringattn_set_bwd_flush_interval(1024)


def test_trace_without_launches(lib):
    """Tracing is host bookkeeping: enabling it and collecting an empty record
    needs no GPU."""
    ra.trace_enable(True)
    assert ra.trace_collect() == {}
    ra.trace_enable(False)
    n = ctypes.c_int(-1)
    assert lib.ringattn_trace_collect(None, -1, ctypes.byref(n)) == -1


def test_rank_step_argument_errors_without_gpu(lib):
    """One ring step of one rank (multi-GPU form): bf16 and the ring exchange
    only, rank and step inside the ring, a workspace for the steps that merge."""
    f = lib.ringattn_fwd_rank_step
    ws = lib.ringattn_fwd_rank_workspace_size(dims(T=256), 2)
    assert ws >= 128 * 2 * 128 * 4 + 2 * 128 * 4
    assert lib.ringattn_bwd_rank_workspace_size(dims(T=256), 2) >= 2 * 128 * 4
    assert f(16, 16, 16, None, dims(dtype=ra.RA_FP32), 2, 0, 1, 0, 0, 16, 16, 16, 16, 16, ws,
             None) == -3
    assert f(16, 16, 16, None, dims(), 2, 0, 1, 2, 0, 16, 16, 16, 16, 16, ws, None) == -1
    assert f(16, 16, 16, None, dims(), 2, 0, 1, 0, 2, 16, 16, 16, 16, 16, ws, None) == -1
    assert f(16, 16, 16, None, dims(T=250), 4, 0, 1, 0, 0, 16, 16, 16, 16, 16, ws, None) == -2
    # a step after the first merges through the workspace
    assert f(16, 16, 16, None, dims(), 2, 0, 1, 0, 1, 16, 16, 16, 16, None, 0, None) == -6
    d = dims()
    d.kv_exchange = 1
    assert f(16, 16, 16, None, d, 2, 0, 1, 0, 0, 16, 16, 16, 16, 16, ws, None) == -3
    b = lib.ringattn_bwd_rank_step
    assert b(16, 16, 16, 16, 16, 16, None, dims(), 2, 0, 1, 0, 0, 16, 16, 16, None, 0,
             None) == -6


def test_debug_library_loads_and_exports_every_symbol():
    """The bounds-checking build exports the same C ABI; its status string
    for a failed check exists."""
    import ctypes as ct
    if not os.path.exists(ra_build.LIB_DEBUG):
        ra_build.build(debug=True)
    dbg = ct.CDLL(ra_build.LIB_DEBUG)
    missing = [n for n in declared_functions() if not hasattr(dbg, n)]
    assert not missing, missing
    dbg.ringattn_status_string.restype = ct.c_char_p
    assert b"bounds" in dbg.ringattn_status_string(-7)
