"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and the fp64 oracle on the same seeded, storage-rounded inputs."""
from __future__ import annotations

import numpy as np

import oracle
from self_attention_backward_gb300 import binding as B

# max|err| / max|ref| per output tensor
TOL = {"f32": 1e-4, "bf16": 2e-2}
TOL_LSE = 1e-4


def rel_err(got, ref) -> float:
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    if den == 0.0:
        return float(np.max(np.abs(got))) if np.size(got) else 0.0
    return float(np.max(np.abs(np.asarray(got, dtype=np.float64) - ref)) / den)


def torch_dtype(dtype: str):
    import torch
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


def to_device(arr: np.ndarray, dtype: str):
    import torch
    # the arrays hold storage-representable values, so this cast is exact
    return torch.from_numpy(np.ascontiguousarray(arr)).to("cuda").to(torch_dtype(dtype)).contiguous()


def gpu_fwd_bwd(inp, algo=B.PSA_ALGO_AUTO):
    """Forward then backward on the GPU; returns fp64 numpy arrays."""
    import torch
    packed = to_device(inp.packed, inp.dtype)
    do_lo = to_device(inp.do_lo, inp.dtype)
    do_hi = to_device(inp.do_hi, inp.dtype)
    o_lo, o_hi, lse = B.attn_fwd(packed, inp.scale)
    d_packed = B.attn_bwd(packed, o_lo, o_hi, lse, do_lo, do_hi, inp.scale, algo=algo)
    B.psa_attn_sync_status()
    torch.cuda.synchronize()
    f = lambda t: t.double().cpu().numpy()  # noqa: E731
    return {"o_lo": f(o_lo), "o_hi": f(o_hi), "lse": f(lse), "d_packed": f(d_packed)}


def oracle_fwd_bwd(inp, slices=None):
    """fp64 oracle on the (storage-rounded) inputs, restricted to `slices`."""
    sl = slice(None) if slices is None else np.asarray(slices)
    p = inp.packed[sl].astype(np.float64)
    vs = np.ascontiguousarray(p[:, 2:4].transpose(1, 0, 2, 3))
    dos = np.stack([inp.do_lo[sl], inp.do_hi[sl]]).astype(np.float64)
    dq, dk, dvs, o, lse, _ = oracle.attn_bwd(p[:, 0], p[:, 1], vs, dos, inp.scale, want_fwd=True)
    return {"o_lo": o[0], "o_hi": o[1], "lse": lse, "d_packed": np.stack([dq, dk, dvs[0], dvs[1]], axis=1)}


SECTIONS = ["dQ", "dK", "dV_lo", "dV_hi"]


def compare(gpu, ref, dtype, slices=None):
    """Per-tensor relative errors; returns {name: err}."""
    sl = slice(None) if slices is None else np.asarray(slices)
    errs = {
        "O_lo": rel_err(gpu["o_lo"][sl], ref["o_lo"]),
        "O_hi": rel_err(gpu["o_hi"][sl], ref["o_hi"]),
        "LSE": rel_err(gpu["lse"][sl], ref["lse"]),
    }
    for s, name in enumerate(SECTIONS):
        errs[name] = rel_err(gpu["d_packed"][sl][:, s], ref["d_packed"][:, s])
    return errs


def assert_within(errs, dtype):
    tol = TOL[dtype]
    bad = {k: v for k, v in errs.items() if v > (TOL_LSE if k == "LSE" else tol) or not np.isfinite(v)}
    assert not bad, f"over tolerance ({dtype}, tol {tol}): {bad}; all: {errs}"
