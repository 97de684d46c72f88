"""Seeded input generator and stored oracle digests (no GPU)."""
import json
import os

import numpy as np
import pytest

from self_attention_backward_gb300.inputs import (WORKLOADS, make_inputs, make_custom, round_bf16)

HERE = os.path.dirname(os.path.abspath(__file__))


def test_round_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(0).normal(size=100000).astype(np.float32) * 37.0
    x[:4] = [1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8, -(1.0 + 2.0**-8), 0.0]  # ties to even
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(round_bf16(x), ref)


def test_generator_is_deterministic_and_shaped():
    a = make_inputs("psa_f32_b1_h2_n16_d16")
    b = make_inputs("psa_f32_b1_h2_n16_d16")
    np.testing.assert_array_equal(a.packed, b.packed)
    np.testing.assert_array_equal(a.do_hi, b.do_hi)
    assert a.packed.shape == (2, 4, 16, 16) and a.do_lo.shape == (2, 16, 16)
    c = make_custom(BH=3, N=7, d=16, dtype="bf16", seed=1)
    assert np.array_equal(c.packed, round_bf16(c.packed))


def test_workload_distributions_small_draw():
    """Moments of a reduced draw of the bf16 N=400 workload: V ~ U(-1,1), dO ~ N(0, 0.1)."""
    inp = make_inputs("psa_bf16_b32_h8_n400_d64", BH=4)
    v = inp.packed[:, 2:4]
    assert v.min() >= -1.0 and v.max() <= 1.0
    assert abs(float(inp.do_lo.std()) - 0.1) < 0.005
    big = make_inputs("psa_bf16_b8_h2_n6400_d32", BH=1, N=512)
    assert abs(float(big.packed[:, 0].std()) - 2.0) < 0.05   # Q ~ N(0, 2): std 2


def test_workload_table():
    assert [w.N for w in WORKLOADS.values()] == [16, 400, 400, 1600, 6400]
    assert [w.BH for w in WORKLOADS.values()] == [2, 32, 256, 64, 16]


@pytest.mark.parametrize("fname", ["psa_f32_b1_h2_n16_d16.json", "ragged_bf16_bh1_n5_d16.json"])
def test_oracle_matches_stored_digest(oracle_mod, fname):
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(HERE, "golden", "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    with open(os.path.join(HERE, "golden", fname)) as f:
        stored = json.load(f)
    now = mg.digest(stored["workload"], mg.CASES[stored["workload"]]())
    for key, t in stored["tensors"].items():
        got = now["tensors"][key]
        for stat in ("sum", "abs_sum", "max_abs"):
            assert got[stat] == pytest.approx(t[stat], rel=1e-12, abs=1e-12), (key, stat)
        for (b, i, c, val), (_, _, _, gv) in zip(t["picks"], got["picks"]):
            assert gv == pytest.approx(val, rel=1e-12, abs=1e-14), (key, b, i, c)
