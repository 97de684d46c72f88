"""Writes the stored oracle values under tests/golden/ (calls only oracle/ and
the seeded input generator).

The pages print no worked example of the attention backward, so nothing here
is a page value: these files record what the fp64 oracle returns on the small
2-slice, N=16, d=16 fp32 workload (seed 0, scale 1/4) and on a ragged N=5 case,
so that a rebuilt oracle on another machine (the Arm GPU host) can be checked
against this one.  What makes the oracle right is pinned in
tests/test_oracle.py; this file only guards against it drifting.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from self_attention_backward_gb300.inputs import make_inputs, make_custom  # noqa: E402

CASES = {
    "psa_f32_b1_h2_n16_d16": lambda: make_inputs("psa_f32_b1_h2_n16_d16"),
    "ragged_bf16_bh1_n5_d16": lambda: make_custom(BH=1, N=5, d=16, dtype="bf16", seed=21),
}
# a few fixed element indices per output tensor (bh, row, col)
PICKS = [(0, 0, 0), (0, 3, 7), (1, 15, 15), (1, 8, 2), (0, 4, 12)]


def digest(name, inp):
    o_lo, o_hi, lse = oracle.psa_fwd(inp.packed, inp.scale)
    dp = oracle.psa_bwd(inp.packed, inp.do_lo, inp.do_hi, inp.scale)
    BH, _, N, d = dp.shape
    out = {"workload": name, "shape": [BH, N, d], "scale": inp.scale, "tensors": {}}
    tens = {"dQ": dp[:, 0], "dK": dp[:, 1], "dV_lo": dp[:, 2], "dV_hi": dp[:, 3],
            "O_lo": o_lo, "O_hi": o_hi, "LSE": lse[..., None]}
    for key, t in tens.items():
        picks = [[b, i, c, float(t[b, i, c])] for b, i, c in PICKS
                 if b < t.shape[0] and i < t.shape[1] and c < t.shape[2]]
        out["tensors"][key] = {"sum": float(t.sum()), "abs_sum": float(np.abs(t).sum()),
                               "max_abs": float(np.abs(t).max()), "picks": picks}
    return out


def main():
    for name, mk in CASES.items():
        with open(os.path.join(HERE, f"{name}.json"), "w") as f:
            json.dump(digest(name, mk()), f, indent=1)
            f.write("\n")


if __name__ == "__main__":
    main()
