"""fp64 CPU oracle for PSA self-attention forward and backward.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package.  It shares no code with
the CUDA library in ``self_attention_backward_gb300`` and imports nothing from
it.

The arithmetic lives in ``psa_oracle.c`` (plain C, fp64, OpenMP over rows); this
module builds it with gcc on first use and marshals numpy arrays through ctypes.
What it computes, and what pins it, is stated in the C file's header: the
definition of softmax attention and its analytic gradient, for ``nv`` V
sections sharing one softmax ("Struct PsaFa2Backward", description and
"Atomicity" paragraphs: lo and hi share Q/K, dQ/dK are summed, each owns dV).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "psa_oracle.c")
_LIB = os.path.join(_HERE, "_psa_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile psa_oracle.c into _psa_oracle.so (gcc, -O2, OpenMP, IEEE fp)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.psa_oracle_fwd.argtypes = [ctypes.c_int] * 4 + [ctypes.c_double] + [_dp] * 5
            lib.psa_oracle_fwd.restype = ctypes.c_int
            lib.psa_oracle_bwd.argtypes = [ctypes.c_int] * 4 + [ctypes.c_double] + [_dp] * 10
            lib.psa_oracle_bwd.restype = ctypes.c_int
            lib.psa_oracle_merge_fwd.argtypes = [ctypes.c_int] * 4 + [_dp] * 3
            lib.psa_oracle_merge_fwd.restype = ctypes.c_int
            lib.psa_oracle_merge_bwd.argtypes = [ctypes.c_int] * 4 + [_dp] * 3
            lib.psa_oracle_merge_bwd.restype = ctypes.c_int
            lib.psa_oracle_threads.argtypes = []
            lib.psa_oracle_threads.restype = ctypes.c_int
            lib.psa_oracle_set_threads.argtypes = [ctypes.c_int]
            lib.psa_oracle_set_threads.restype = None
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(_dp)


def threads() -> int:
    """OpenMP threads the oracle runs with."""
    return int(_load().psa_oracle_threads())


def set_threads(n: int) -> None:
    _load().psa_oracle_set_threads(int(n))


def attn_fwd(q, k, vs, scale: float):
    """Forward for nv V sections sharing one softmax.

    q, k: [BH, N, d]; vs: [nv, BH, N, d].  Returns (o [nv, BH, N, d], lse [BH, N]).
    """
    q, k, vs = _f64(q), _f64(k), _f64(vs)
    nv, BH, N, d = vs.shape
    assert q.shape == (BH, N, d) and k.shape == (BH, N, d)
    o = np.empty((nv, BH, N, d))
    lse = np.empty((BH, N))
    rc = _load().psa_oracle_fwd(BH, N, d, nv, float(scale), _ptr(q), _ptr(k), _ptr(vs), _ptr(o), _ptr(lse))
    if rc:
        raise RuntimeError(f"psa_oracle_fwd failed ({rc})")
    return o, lse


def attn_bwd(q, k, vs, dos, scale: float, want_fwd: bool = False):
    """Backward for nv V sections sharing one softmax.

    q, k: [BH, N, d]; vs, dos: [nv, BH, N, d].
    Returns (dq, dk, dvs) -- and (o, lse, D) too when ``want_fwd``.
    """
    q, k, vs, dos = _f64(q), _f64(k), _f64(vs), _f64(dos)
    nv, BH, N, d = vs.shape
    assert dos.shape == vs.shape and q.shape == (BH, N, d) and k.shape == (BH, N, d)
    dq = np.empty((BH, N, d))
    dk = np.empty((BH, N, d))
    dvs = np.empty((nv, BH, N, d))
    o = np.empty((nv, BH, N, d)) if want_fwd else None
    lse = np.empty((BH, N)) if want_fwd else None
    D = np.empty((BH, N)) if want_fwd else None
    rc = _load().psa_oracle_bwd(BH, N, d, nv, float(scale), _ptr(q), _ptr(k), _ptr(vs), _ptr(dos),
                                _ptr(dq), _ptr(dk), _ptr(dvs), _ptr(o), _ptr(lse), _ptr(D))
    if rc:
        raise RuntimeError(f"psa_oracle_bwd failed ({rc})")
    if want_fwd:
        return dq, dk, dvs, o, lse, D
    return dq, dk, dvs


def psa_fwd(packed, scale: float):
    """PSA forward on a packed [BH, 4, N, d] buffer (sections Q, K, V_lo, V_hi).

    Returns (o_lo, o_hi, lse) with o_* [BH, N, d] and lse [BH, N].
    """
    packed = _f64(packed)
    vs = np.ascontiguousarray(packed[:, 2:4].transpose(1, 0, 2, 3))
    o, lse = attn_fwd(packed[:, 0], packed[:, 1], vs, scale)
    return o[0], o[1], lse


def psa_bwd(packed, do_lo, do_hi, scale: float):
    """PSA backward on a packed [BH, 4, N, d] buffer.

    Returns d_packed [BH, 4, N, d]: sections dQ, dK (summed over lo and hi),
    dV_lo, dV_hi.
    """
    packed = _f64(packed)
    vs = np.ascontiguousarray(packed[:, 2:4].transpose(1, 0, 2, 3))
    dos = np.stack([_f64(do_lo), _f64(do_hi)])
    dq, dk, dvs = attn_bwd(packed[:, 0], packed[:, 1], vs, dos, scale)
    return np.stack([dq, dk, dvs[0], dvs[1]], axis=1)


def merge_fwd(o_lo, o_hi, B: int, heads: int):
    """PSA attention merge ("Struct PsaMergeAttnRuntimeOp"): O_lo, O_hi
    [B*heads, N, d] -> merged [B, 2*heads*d, N], lo in the low half of the
    channels and hi in the high half, head-major in each (the reading stated in
    psa_oracle.c)."""
    o_lo, o_hi = _f64(o_lo), _f64(o_hi)
    BH, N, d = o_lo.shape
    assert BH == B * heads and o_hi.shape == o_lo.shape
    out = np.empty((B, 2 * heads * d, N))
    if _load().psa_oracle_merge_fwd(B, heads, N, d, _ptr(o_lo), _ptr(o_hi), _ptr(out)):
        raise RuntimeError("psa_oracle_merge_fwd failed")
    return out


def merge_bwd(d_merged, heads: int, d: int):
    """The merge's backward: d_merged [B, 2*heads*d, N] -> (dO_lo, dO_hi), each
    [B*heads, N, d]."""
    g = _f64(d_merged)
    B, c, N = g.shape
    assert c == 2 * heads * d
    d_lo = np.empty((B * heads, N, d))
    d_hi = np.empty((B * heads, N, d))
    if _load().psa_oracle_merge_bwd(B, heads, N, d, _ptr(g), _ptr(d_lo), _ptr(d_hi)):
        raise RuntimeError("psa_oracle_merge_bwd failed")
    return d_lo, d_hi
