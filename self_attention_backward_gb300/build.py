"""Builds the CUDA library ``_psa_attn.so`` in-tree for sm_103a (nvcc only).

Each translation unit under ``csrc/`` is compiled in parallel with
``-gencode arch=compute_103a,code=sm_103a``, then linked into one shared
library with a plain C ABI (``include/psa_attn.h``).

    python -m self_attention_backward_gb300.build
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "_psa_attn.so")
BUILD_DIR = os.path.join(PKG, "_build")
SOURCES = ["psa_attn.cu", "tc_bwd.cu", "tc_fwd.cu", "noalloc.cu", "tc_dq.cu", "tc_pair.cu", "tc_tmap.cu", "host_pipe.cu",
           "merge.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                   "--expt-relaxed-constexpr", *extra]


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "psa_attn.h"))
    objs, procs = [], []
    for src in SOURCES:
        sp = os.path.join(CSRC, src)
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [sp, *headers, __file__]):
            cmd = [_nvcc(), *_flags(extra_flags), "-c", sp, "-o", obj]
            if verbose:
                print(" ".join(cmd), flush=True)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    errors = []
    for src, p in procs:
        out, _ = p.communicate()
        if out and (verbose or p.returncode):
            sys.stdout.write(out.decode(errors="replace"))
        if p.returncode:
            errors.append(src)
    if errors:
        raise RuntimeError(f"nvcc failed for {errors}")
    if force or procs or _stale(LIB, objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
