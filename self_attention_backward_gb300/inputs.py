"""Seeded synthetic inputs for PSA self-attention (shared by the oracle side and
the CUDA side; holds none of the attention arithmetic).

Workloads are PSA attention blocks of a YOLO-style detector: one (batch, head)
slice attends over the N = H*W positions of a feature map.  Each slice owns a
packed buffer of four [N, d] sections in the order Q, K, V_lo, V_hi, and the
upstream gradients dO_lo, dO_hi are [N, d] each.  The pages benchmark on no
dataset; these synthetic tensors have the shapes and value distributions of
the five workloads below.

Draw order for a workload with seed s (numpy ``default_rng(s)``, float64
draws, one call per section, each section shaped [BH, N, d]):
    Q, K, V_lo, V_hi, dO_lo, dO_hi
Normal distributions are given as (mean, standard deviation).  Values are then
rounded float64 -> float32 -> storage type (bf16 by round-to-nearest-even).
"""
from __future__ import annotations

from dataclasses import dataclass, field
import math

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "f32" or "bf16" storage; accumulation is always fp32
    B: int
    heads: int
    N: int
    d: int
    seed: int
    scale: float
    # distribution per section: ("normal", mean, std) or ("uniform", lo, hi)
    q: tuple = ("normal", 0.0, 1.0)
    k: tuple = ("normal", 0.0, 1.0)
    v: tuple = ("normal", 0.0, 1.0)
    do: tuple = ("normal", 0.0, 1.0)
    fmap: str = ""

    @property
    def BH(self) -> int:
        return self.B * self.heads


WORKLOADS = {
    w.name: w
    for w in [
        Workload("psa_f32_b1_h2_n16_d16", "f32", 1, 2, 16, 16, 0, 1.0 / math.sqrt(16), fmap="4x4"),
        Workload("psa_f32_b8_h4_n400_d64", "f32", 8, 4, 400, 64, 1, 1.0 / 8, fmap="20x20"),
        Workload("psa_bf16_b32_h8_n400_d64", "bf16", 32, 8, 400, 64, 2, 1.0 / 8,
                 v=("uniform", -1.0, 1.0), do=("normal", 0.0, 0.1), fmap="20x20"),
        Workload("psa_bf16_b16_h4_n1600_d64", "bf16", 16, 4, 1600, 64, 3, 1.0 / 8, fmap="40x40"),
        Workload("psa_bf16_b8_h2_n6400_d32", "bf16", 8, 2, 6400, 32, 4, 1.0 / math.sqrt(32),
                 q=("normal", 0.0, 2.0), k=("normal", 0.0, 2.0), fmap="80x80"),
    ]
}
WORKLOAD_ORDER = list(WORKLOADS)


def _draw(rng: np.random.Generator, dist: tuple, shape) -> np.ndarray:
    kind, a, b = dist
    if kind == "normal":
        return rng.normal(a, b, size=shape)
    if kind == "uniform":
        return rng.uniform(a, b, size=shape)
    raise ValueError(f"unknown distribution {kind!r}")


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns
    float32 holding bf16-representable values.  Inputs are finite."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def round_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    x32 = np.asarray(x, dtype=np.float32)
    if dtype == "f32":
        return np.ascontiguousarray(x32)
    if dtype == "bf16":
        return round_bf16(x32)
    raise ValueError(dtype)


@dataclass
class Inputs:
    """Storage-rounded inputs as float32 numpy arrays."""
    packed: np.ndarray     # [BH, 4, N, d]: Q, K, V_lo, V_hi
    do_lo: np.ndarray      # [BH, N, d]
    do_hi: np.ndarray      # [BH, N, d]
    dtype: str
    scale: float
    extra: dict = field(default_factory=dict)


def make_inputs(w: Workload | str, *, BH: int | None = None, N: int | None = None,
                d: int | None = None, seed: int | None = None) -> Inputs:
    """Draw one workload's inputs.  BH / N / d / seed may be overridden to get a
    smaller case with the same distributions."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    BH = w.BH if BH is None else BH
    N = w.N if N is None else N
    d = w.d if d is None else d
    seed = w.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    shape = (BH, N, d)
    secs = [_draw(rng, dist, shape) for dist in (w.q, w.k, w.v, w.v)]
    do_lo = _draw(rng, w.do, shape)
    do_hi = _draw(rng, w.do, shape)
    packed = np.stack(secs, axis=1)
    return Inputs(
        packed=round_storage(packed, w.dtype),
        do_lo=round_storage(do_lo, w.dtype),
        do_hi=round_storage(do_hi, w.dtype),
        dtype=w.dtype,
        scale=float(w.scale),
    )


def make_custom(BH: int, N: int, d: int, dtype: str, seed: int, scale: float | None = None,
                q=("normal", 0.0, 1.0), k=("normal", 0.0, 1.0), v=("normal", 0.0, 1.0),
                do=("normal", 0.0, 1.0)) -> Inputs:
    """Inputs of an arbitrary shape (ragged and edge cases)."""
    w = Workload("custom", dtype, 1, BH, N, d, seed,
                 scale if scale is not None else 1.0 / math.sqrt(d), q=q, k=k, v=v, do=do)
    return make_inputs(w)
