"""Builds libringattn.so in-tree with nvcc for sm_103a (B300).

    python -m context_long_sequence_fwd_b300.build [--force] [--debug] [-v]

Objects go to ``_build/`` next to this file; the shared library is written
to ``context_long_sequence_fwd_b300/libringattn.so`` (the binding loads it
from there).  ``--debug`` builds the bounds-checking variant (RINGATTN_DEBUG:
every kernel checks the global indices it computes) into ``_build_debug/``
and ``libringattn_debug.so``, which the binding loads when the environment
sets RINGATTN_DEBUG=1.  nvcc cross-compiles, so no GPU is needed to build.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libringattn.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libringattn_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
          "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build")
    return path


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cu", ".cpp")))


def headers() -> list[str]:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _mtime(p: str) -> float:
    return os.path.getmtime(p) if os.path.exists(p) else -1.0


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    newest_header = max((_mtime(h) for h in headers()), default=0.0)
    flags = list(COMMON) + (["-DRINGATTN_DEBUG"] if debug else [])
    jobs = []
    for src in sources():
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        if force or _mtime(obj) < max(_mtime(src), newest_header):
            cmd = [nvcc()] + ARCH + flags + ["-Xptxas", "-v", "-c", src, "-o", obj]
            jobs.append((src, obj, cmd))
    objs = [os.path.join(build_dir, os.path.basename(s) + ".o") for s in sources()]

    def run(job):
        src, obj, cmd = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, r

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
            for src, r in ex.map(run, jobs):
                if r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                    raise RuntimeError(f"nvcc failed on {os.path.basename(src)}")
                if verbose:
                    sys.stderr.write(r.stderr)
    if force or jobs or _mtime(lib) < max(_mtime(o) for o in objs):
        tmp = lib + f".{os.getpid()}.tmp"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError(f"link of {os.path.basename(lib)} failed")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    ap.add_argument("--debug", action="store_true", help="the bounds-checking build")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, debug=a.debug))
