"""The oracle's pins must catch plausible mistakes.

Each case copies the oracle's C source, plants one mistake in the copy (a
dropped term, a wrong sign, an off-by-one mask, a wrong operand or head
index), builds it into a temporary library and runs the pins against it: at
least one pin must fail.  The real oracle is never modified.
"""
import contextlib
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle as pins
from tests import test_oracle_ssd as ssd_pins

HERE = os.path.dirname(oracle.__file__)
SRC = os.path.join(HERE, "attention_fp64.c")
SSD_SRC = os.path.join(HERE, "ssd_fp64.c")

MUTANTS = {
    "causal_excludes_diagonal": ("if (causal && j > i) return 0;",
                                 "if (causal && j >= i) return 0;"),
    "lse_drops_max": ("return m + log(z);", "return log(z);"),
    "no_scale": ("s[j] = p->scale * dot(qi, kj, p->d);",
                 "s[j] = dot(qi, kj, p->d);"),
    "gqa_wrong_head": ("    int g = h / group;\n    const double *qi",
                       "    int g = h % p->hkv;\n    const double *qi"),
    "doc_bound_inclusive": ("t < cu_seqlens[d + 1]", "t <= cu_seqlens[d + 1]"),
    "dS_wrong_sign": ("double dS = P * (dot(doi, vj, d) - D);",
                      "double dS = P * (dot(doi, vj, d) + D);"),
    "dq_no_scale": ("dq_row[c] += p->scale * dS * kj[c];",
                    "dq_row[c] += dS * kj[c];"),
    "dv_wrong_operand": ("dvr[c] += P * doi[c];", "dvr[c] += P * qi[c];"),
    "dk_drops_D": ("double dS = P * (dot(doi, vj, d) - Dv[(size_t)h * T + i]);",
                   "double dS = P * dot(doi, vj, d);"),
    "merge_weights_swapped": ("double wa = exp(a - L), wb = exp(b - L);",
                              "double wa = exp(b - L), wb = exp(a - L);"),
    "merge_empty_side": ("if (b == -INFINITY) continue;",
                         "if (b == -INFINITY) { lse_a[r] = b; continue; }"),
}


SSD_MUTANTS = {
    "ssd_decay_without_dt": ("double a = exp(d * A[h]);", "double a = exp(A[h]);"),
    "ssd_input_without_dt": ("Sp[n] = a * Sp[n] + d * xt[p] * Bt[n];",
                             "Sp[n] = a * Sp[n] + xt[p] * Bt[n];"),
    "ssd_no_reset": ("if (pos && pos[t] == 0) memset", "if (pos && pos[t] == -1) memset"),
    "ssd_reads_B_for_C": ("acc += Sp[n] * Ct[n];", "acc += Sp[n] * Bt[n];"),
    "ssd_drops_skip": ("yt[p] = acc + (D ? D[h] : 0.0) * xt[p];", "yt[p] = acc;"),
    "ssd_output_before_update": (
        "Sp[n] = a * Sp[n] + d * xt[p] * Bt[n];\n                    acc += Sp[n] * Ct[n];",
        "acc += Sp[n] * Ct[n];\n                    Sp[n] = a * Sp[n] + d * xt[p] * Bt[n];"),
    "ssd_group_of_head": ("int g = h / per_group;", "int g = h % G;"),
}


@contextlib.contextmanager
def mutant_oracle(tmp_path, name):
    ssd = name in SSD_MUTANTS
    old, new = SSD_MUTANTS[name] if ssd else MUTANTS[name]
    target = SSD_SRC if ssd else SRC
    src = open(target).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    other = SRC if ssd else SSD_SRC
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                    "-o", str(so), str(path), other, "-lm"], check=True)
    real = oracle._load()
    lib = ctypes.CDLL(str(so))
    for fn in ("oracle_fwd_rows", "oracle_bwd_rows", "oracle_bwd_keys",
               "oracle_lse_merge", "oracle_num_threads", "oracle_ssd_scan"):
        getattr(lib, fn).argtypes = getattr(real, fn).argtypes
        getattr(lib, fn).restype = getattr(real, fn).restype
    oracle._lib = lib
    try:
        yield
    finally:
        oracle._lib = real


@pytest.mark.parametrize("name", list(MUTANTS) + list(SSD_MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    failed = []
    suite = ssd_pins.PINS if name in SSD_MUTANTS else pins.PINS
    with mutant_oracle(tmp_path, name):
        for pin_name, fn in suite.items():
            try:
                fn()
            except AssertionError:
                failed.append(pin_name)
    assert failed, f"no pin caught mutant {name}"
