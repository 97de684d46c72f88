"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded, storage-rounded inputs.  Tolerance per output tensor:
max|err| / max|ref| <= 1e-4 for fp32 storage, <= 2e-2 for bf16 storage
(LSE, always fp32, <= 1e-4)."""
import numpy as np
import pytest

from self_attention_backward_gb300 import binding as B
from self_attention_backward_gb300.inputs import WORKLOADS, make_inputs, make_custom

from gpu_helpers import assert_within, compare, gpu_fwd_bwd, oracle_fwd_bwd, rel_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from self_attention_backward_gb300.build import build
    build()


def algos_for(dtype, d):
    out = [B.PSA_ALGO_SIMT]
    if B.psa_attn_bwd_workspace_bytes(1, 1, 16, d, {"f32": 0, "bf16": 1}[dtype], B.PSA_ALGO_TC) > 0:
        out += [B.PSA_ALGO_TC, B.PSA_ALGO_TC_2PASS]
    return out


# Full-size workloads in the launch configuration the bench times; the oracle
# checks the listed (batch*head) slices, which it computes one by one.  On a
# 152-SM GPU the fused mode splits the last wave's units along the queries:
# at N=1600 those are the key tiles 6-12 of slice 58 and all of slices 59-63,
# at N=6400 the key tiles 10-49 of slice 15; the samples include both.
SAMPLED = {
    "psa_f32_b1_h2_n16_d16": None,
    "psa_f32_b8_h4_n400_d64": None,
    "psa_bf16_b32_h8_n400_d64": [0, 101, 200, 255],
    "psa_bf16_b16_h4_n1600_d64": [0, 37, 58, 63],
    "psa_bf16_b8_h2_n6400_d32": [0, 5, 10, 15],
}
# per-block bound: a block's max|err| against its own max|ref|
BLOCK_TOL_MUL = 3.0

_oracle_cache = {}


def _ref(name):
    if name not in _oracle_cache:
        inp = make_inputs(name)
        _oracle_cache[name] = (inp, oracle_fwd_bwd(inp, SAMPLED[name]))
    return _oracle_cache[name]


@pytest.mark.parametrize("name", list(SAMPLED))
@pytest.mark.parametrize("algo", [B.PSA_ALGO_SIMT, B.PSA_ALGO_TC, B.PSA_ALGO_TC_2PASS])
def test_workload_parity(name, algo):
    w = WORKLOADS[name]
    if algo not in algos_for(w.dtype, w.d):
        pytest.skip("no tensor-core kernel for this dtype/head_dim")
    inp, ref = _ref(name)
    gpu = gpu_fwd_bwd(inp, algo)
    errs = compare(gpu, ref, inp.dtype, SAMPLED[name])
    print(name, algo, errs)
    assert_within(errs, inp.dtype)
    check_blocks(gpu["d_packed"], ref["d_packed"], inp.dtype, SAMPLED[name])


def check_blocks(got, ref, dtype, slices=None):
    """Every 64-query block of dQ and every 128-key block of dK, dV_lo and dV_hi
    of every checked slice against the oracle, each against its own max|ref|:
    one bad tile cannot hide under the whole tensor's maximum."""
    from gpu_helpers import TOL
    rows = range(ref.shape[0]) if slices is None else range(len(slices))
    N = ref.shape[2]
    for k in rows:
        g = got[k] if slices is None else got[slices[k]]
        r = ref[k]
        for q0 in range(0, N, 64):
            blk = slice(q0, min(N, q0 + 64))
            e = rel_err(g[0, blk], r[0, blk])
            assert e < BLOCK_TOL_MUL * TOL[dtype], ("dQ", k, q0, e)
        for k0 in range(0, N, 128):
            blk = slice(k0, min(N, k0 + 128))
            for sec in (1, 2, 3):
                e = rel_err(g[sec, blk], r[sec, blk])
                assert e < BLOCK_TOL_MUL * TOL[dtype], (sec, k, k0, e)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("N", [1, 17, 127, 129, 400])
def test_ragged_parity(N, d, dtype):
    inp = make_custom(BH=3, N=N, d=d, dtype=dtype, seed=1000 + N + d)
    ref = oracle_fwd_bwd(inp)
    for algo in algos_for(dtype, d):
        errs = compare(gpu_fwd_bwd(inp, algo), ref, dtype)
        assert_within(errs, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_equal_v_rows_give_zero_dq_dk(dtype):
    """Every row of V_lo equal and every row of V_hi equal: dS = 0, so dQ = dK = 0
    up to rounding, while dV stays O(1)."""
    inp = make_custom(BH=2, N=129, d=64, dtype=dtype, seed=77)
    inp.packed[:, 2] = inp.packed[:, 2, :1]
    inp.packed[:, 3] = inp.packed[:, 3, :1]
    for algo in algos_for(dtype, 64):
        g = gpu_fwd_bwd(inp, algo)["d_packed"]
        dv = np.max(np.abs(g[:, 2:4]))
        assert dv > 0.1
        assert np.max(np.abs(g[:, 0:2])) < (1e-4 if dtype == "f32" else 2e-2) * dv


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_dv_sums_match_do_sums(dtype):
    """Rows of P sum to 1: sum over keys of dV_h equals sum over queries of dO_h."""
    inp = make_custom(BH=2, N=400, d=32, dtype=dtype, seed=78)
    for algo in algos_for(dtype, 32):
        g = gpu_fwd_bwd(inp, algo)["d_packed"]
        for h, do in ((2, inp.do_lo), (3, inp.do_hi)):
            ref = do.astype(np.float64).sum(axis=1)
            assert rel_err(g[:, h].sum(axis=1), ref) < (1e-4 if dtype == "f32" else 2e-2)


@pytest.mark.parametrize("algo", [B.PSA_ALGO_SIMT, B.PSA_ALGO_TC_2PASS])
def test_atomic_free_modes_are_deterministic(algo):
    """The CUDA-core and two-pass tensor-core backwards sum every output in a
    fixed order: repeated runs agree bit for bit (many key and query tiles, a
    ragged tail)."""
    for d in (16, 32, 64):
        inp = make_custom(BH=3, N=777, d=d, dtype="bf16", seed=79 + d)
        a = gpu_fwd_bwd(inp, algo)["d_packed"]
        for _ in range(2):
            np.testing.assert_array_equal(a, gpu_fwd_bwd(inp, algo)["d_packed"])


@pytest.mark.parametrize("d", [16, 32, 64])
def test_two_pass_matches_fused_tensor_core(d):
    """The two tensor-core modes compute the same products with the same bf16
    roundings of P and dS; they differ only in fp32 summation order."""
    inp = make_custom(BH=2, N=1000, d=d, dtype="bf16", seed=90 + d)
    a = gpu_fwd_bwd(inp, B.PSA_ALGO_TC)["d_packed"]
    b = gpu_fwd_bwd(inp, B.PSA_ALGO_TC_2PASS)["d_packed"]
    for sec in range(4):
        assert rel_err(b[:, sec], a[:, sec]) < 1e-2, sec


def test_overwrites_d_packed_and_stream_arg():
    """d_packed is overwritten (not accumulated), and an explicit side stream works."""
    inp = make_custom(BH=2, N=65, d=16, dtype="f32", seed=80)
    from gpu_helpers import to_device
    packed = to_device(inp.packed, "f32")
    do_lo, do_hi = to_device(inp.do_lo, "f32"), to_device(inp.do_hi, "f32")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o_lo, o_hi, lse = B.attn_fwd(packed, inp.scale)
        garbage = torch.full_like(packed, 1e30)
        out = B.attn_bwd(packed, o_lo, o_hi, lse, do_lo, do_hi, inp.scale, d_packed=garbage)
    s.synchronize()
    ref = oracle_fwd_bwd(inp)["d_packed"]
    assert rel_err(out.double().cpu().numpy(), ref) < 1e-4


def test_sync_status_ok():
    assert B.psa_attn_sync_status() == 0


def test_bounded_wait_timeout_is_reported_and_context_survives():
    """A device-side wait that nothing satisfies gives up after its limit and
    is reported as PSA_ERR_TIMEOUT by psa_attn_sync_status; the context stays
    usable and the flag is cleared."""
    assert B.psa_attn_sync_status() == 0
    B.psa_attn_selftest_wait_timeout()
    rc = B.psa_attn_sync_status(check=False)
    assert rc == B.PSA_ERR_TIMEOUT, (rc, B.psa_attn_last_error())
    assert "gave up" in B.psa_attn_last_error()
    assert B.psa_attn_sync_status() == 0        # cleared
    inp = make_custom(BH=1, N=70, d=32, dtype="bf16", seed=81)
    errs = compare(gpu_fwd_bwd(inp, B.PSA_ALGO_TC), oracle_fwd_bwd(inp), "bf16")
    assert_within(errs, "bf16")


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("N", [1, 100, 128, 300])
def test_tensor_core_forward_matches_oracle(N, d):
    """The tensor-core forward (bf16) against the oracle's O and LSE, and the
    CUDA-core forward on the same inputs."""
    import torch
    from gpu_helpers import to_device, TOL, TOL_LSE
    inp = make_custom(BH=3, N=N, d=d, dtype="bf16", seed=2000 + N + d)
    ref = oracle_fwd_bwd(inp)
    packed = to_device(inp.packed, "bf16")
    for algo in (B.PSA_ALGO_TC, B.PSA_ALGO_SIMT):
        o_lo, o_hi, lse = B.attn_fwd(packed, inp.scale, algo=algo)
        B.psa_attn_sync_status()
        assert rel_err(o_lo.double().cpu().numpy(), ref["o_lo"]) <= TOL["bf16"]
        assert rel_err(o_hi.double().cpu().numpy(), ref["o_hi"]) <= TOL["bf16"]
        assert rel_err(lse.double().cpu().numpy(), ref["lse"]) <= TOL_LSE


def test_tensor_core_forward_full_size_sampled():
    """Tensor-core forward at the N=6400, d=32 workload size (sampled slices)."""
    from gpu_helpers import to_device, TOL, TOL_LSE
    inp = make_inputs("psa_bf16_b8_h2_n6400_d32")
    ref = oracle_fwd_bwd(inp, [3])
    packed = to_device(inp.packed, "bf16")
    o_lo, o_hi, lse = B.attn_fwd(packed, inp.scale, algo=B.PSA_ALGO_TC)
    B.psa_attn_sync_status()
    assert rel_err(o_lo[3].double().cpu().numpy(), ref["o_lo"][0]) <= TOL["bf16"]
    assert rel_err(o_hi[3].double().cpu().numpy(), ref["o_hi"][0]) <= TOL["bf16"]
    assert rel_err(lse[3].double().cpu().numpy(), ref["lse"][0]) <= TOL_LSE


@pytest.mark.parametrize("chunks", [None, 1, 3, 6])
def test_host_buffers_pipelined_match_device_path(chunks):
    """psa_attn_bwd_host through HostBwd (host tensors in, host d_packed out,
    slices pipelined over streams in `chunks` groups, None = the library's
    choice) gives the device path's result: bit for bit in the two-pass mode,
    and within tolerance of the oracle."""
    import torch
    from gpu_helpers import to_device, TOL
    inp = make_custom(BH=6, N=132, d=32, dtype="bf16", seed=95)
    dev = gpu_fwd_bwd(inp, B.PSA_ALGO_TC_2PASS)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).pin_memory()  # noqa: E731
    packed, do_lo, do_hi = pin(inp.packed), pin(inp.do_lo), pin(inp.do_hi)
    o_lo, o_hi, lse = B.attn_fwd(to_device(inp.packed, "bf16"), inp.scale)
    o_lo, o_hi, lse = o_lo.cpu().pin_memory(), o_hi.cpu().pin_memory(), lse.cpu().pin_memory()
    out = torch.empty(packed.shape, dtype=torch.bfloat16).pin_memory()
    runner = B.HostBwd(6, 132, 32, B.PSA_BF16, algo=B.PSA_ALGO_TC_2PASS, chunks=chunks)
    for _ in range(2):  # the second call reuses the staging buffers
        runner(packed, o_lo, o_hi, lse, do_lo, do_hi, inp.scale, out)
    torch.cuda.synchronize()
    B.psa_attn_sync_status()
    got = out.double().numpy()
    np.testing.assert_array_equal(got, dev["d_packed"])
    ref = oracle_fwd_bwd(inp)["d_packed"]
    assert rel_err(got, ref) < TOL["bf16"]


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("algo", [B.PSA_ALGO_TC, B.PSA_ALGO_TC_2PASS])
def test_tensor_core_many_subtiles_repeated(d, algo):
    """Every tensor-core mode on inputs with many key and query tiles (N = 1000
    and 1537: 16 and 25 sub-tiles of 64 queries, ragged), three seeds, three
    runs each, all against the oracle: a scheduling-dependent hazard between
    pipeline stages would show up as a run or a sub-tile out of tolerance."""
    from gpu_helpers import TOL
    for N, seed in ((1000, 301), (1537, 302), (1000, 303)):
        inp = make_custom(BH=2, N=N, d=d, dtype="bf16", seed=seed + d)
        ref = oracle_fwd_bwd(inp)
        for _ in range(3):
            g = gpu_fwd_bwd(inp, algo)["d_packed"]
            for sec in range(4):
                err = rel_err(g[:, sec], ref["d_packed"][:, sec])
                assert err < TOL["bf16"], (N, seed, sec, err)
                # and per 64-query block of dQ (a single bad sub-tile stands out)
            for q0 in range(0, N, 64):
                blk = slice(q0, min(N, q0 + 64))
                assert rel_err(g[:, 0, blk], ref["d_packed"][:, 0, blk]) < 3 * TOL["bf16"], (N, seed, q0)


@pytest.mark.parametrize("dtype,d", [("bf16", 16), ("bf16", 32), ("bf16", 64), ("f32", 32)])
def test_negative_scale(dtype, d):
    """The scale is any finite number: with a negative one the softmax favours
    the smallest q.k.  Forward and every backward family against the oracle."""
    import dataclasses
    inp = make_custom(BH=2, N=300, d=d, dtype=dtype, seed=400 + d)
    inp = dataclasses.replace(inp, scale=-inp.scale)
    ref = oracle_fwd_bwd(inp)
    for algo in algos_for(dtype, d):
        errs = compare(gpu_fwd_bwd(inp, algo), ref, dtype)
        assert_within(errs, dtype)


@pytest.mark.parametrize("dtype,d", [("bf16", 32), ("bf16", 64), ("f32", 16)])
def test_zero_scale_is_uniform_attention(dtype, d):
    """scale = 0: P is uniform (1/N per key), so dQ = dK = 0, every dV_h row is
    the mean of dO_h over the queries, O_h rows are the mean of V_h and
    LSE = log N.  Every kernel family that supports the case."""
    import dataclasses
    from gpu_helpers import TOL
    inp = dataclasses.replace(make_custom(BH=2, N=193, d=d, dtype=dtype, seed=500 + d), scale=0.0)
    tol = TOL[dtype]
    for algo in algos_for(dtype, d):
        g = gpu_fwd_bwd(inp, algo)
        assert np.allclose(g["lse"], np.log(193.0), rtol=1e-5)
        dp = g["d_packed"]
        assert np.max(np.abs(dp[:, 0:2])) == 0.0, algo
        for h, do in ((2, inp.do_lo), (3, inp.do_hi)):
            mean = do.astype(np.float64).mean(axis=1, keepdims=True)      # [BH, 1, d]
            assert rel_err(dp[:, h], np.broadcast_to(mean, dp[:, h].shape)) < tol, (algo, h)


def test_many_slices_large_grid():
    """B*heads = 70001 with N = 16: one-dimensional grids of more than 65535
    CTAs on every kernel family; sampled slices (first, middle, last) against
    the oracle."""
    inp = make_custom(BH=70001, N=16, d=32, dtype="bf16", seed=600)
    slices = [0, 35000, 70000]
    ref = oracle_fwd_bwd(inp, slices)
    for algo in algos_for("bf16", 32):
        errs = compare(gpu_fwd_bwd(inp, algo), ref, "bf16", slices)
        assert_within(errs, "bf16")


@pytest.mark.parametrize("BH,N,d,slices", [
    (1, 900, 32, None),      # 8 units, each split into 8 one-group pieces; last piece one sub-tile
    (3, 700, 64, None),      # 18 units, 6 pieces each
    (2, 1537, 16, None),     # 26 units, 5 pieces of 2-3 groups
    (20, 1000, 32, [0, 19]),  # 160 units on 152 SMs: 152 whole units, the last 8 split
])
def test_fused_query_split_of_last_wave(BH, N, d, slices):
    """The fused tensor-core mode splits the units (batch*head, 128-key tile)
    of its last, partial wave along the query axis and sums the pieces' dK/dV
    partials afterwards.  Shapes whose unit counts make it split (on a
    152-SM GPU) into 1-group pieces, ragged pieces and a mix of whole and split
    units; every section per 128-key block against the oracle."""
    from gpu_helpers import TOL
    inp = make_custom(BH=BH, N=N, d=d, dtype="bf16", seed=700 + d + BH)
    ref = oracle_fwd_bwd(inp, slices)
    g = gpu_fwd_bwd(inp, B.PSA_ALGO_TC)["d_packed"]
    rows = slices if slices is not None else list(range(BH))
    for k, bh in enumerate(rows):
        r = ref["d_packed"][k] if slices is not None else ref["d_packed"][bh]
        for sec in range(4):
            assert rel_err(g[bh, sec], r[sec]) < TOL["bf16"], (bh, sec)
        for k0 in range(0, N, 128):
            blk = slice(k0, min(N, k0 + 128))
            for sec in (1, 2, 3):
                assert rel_err(g[bh, sec, blk], r[sec, blk]) < 3 * TOL["bf16"], (bh, sec, k0)


@pytest.mark.parametrize("N,chunks", [(130, 3), (6400, None)])
def test_host_entry_fused_mode(N, chunks):
    """psa_attn_bwd_host in the fused tensor-core mode: N = 130 (N % 4 != 0,
    so one chunk whatever is asked) and the N = 6400, d = 32 shape with four
    slices and the library's chunk choice; against the oracle (sampled slices
    at N = 6400)."""
    import torch
    from gpu_helpers import TOL
    BH = 4
    inp = make_custom(BH=BH, N=N, d=32, dtype="bf16", seed=97 + N)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).pin_memory()  # noqa: E731
    packed, do_lo, do_hi = pin(inp.packed), pin(inp.do_lo), pin(inp.do_hi)
    o_lo, o_hi, lse = B.attn_fwd(packed.cuda(), inp.scale)
    o_lo, o_hi, lse = o_lo.cpu().pin_memory(), o_hi.cpu().pin_memory(), lse.cpu().pin_memory()
    out = torch.full(packed.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    runner = B.HostBwd(BH, N, 32, B.PSA_BF16, algo=B.PSA_ALGO_TC, chunks=chunks)
    runner(packed, o_lo, o_hi, lse, do_lo, do_hi, inp.scale, out)
    torch.cuda.synchronize()
    B.psa_attn_sync_status()
    slices = [0, BH - 1] if N > 1000 else None
    ref = oracle_fwd_bwd(inp, slices)["d_packed"]
    got = out.double().numpy()
    got = got[slices] if slices else got
    assert np.isfinite(got).all()
    assert rel_err(got, ref) < TOL["bf16"]


@pytest.mark.parametrize("algo", [B.PSA_ALGO_TC, B.PSA_ALGO_TC_2PASS])
@pytest.mark.parametrize("N", [65, 129, 193])
def test_head_dim_16_first_subtiles(N, algo):
    """head_dim 16 with 2-4 query sub-tiles: the first sub-tiles' S/dP products
    are issued before any softmax has run, while the first softmax reads its
    buffer.  Five seeds, three runs each; every 64-query block of dQ and every
    128-key block of dK/dV against the oracle."""
    for seed in range(5):
        inp = make_custom(BH=3, N=N, d=16, dtype="bf16", seed=3100 + 7 * N + seed)
        ref = oracle_fwd_bwd(inp)
        for _ in range(3):
            g = gpu_fwd_bwd(inp, algo)
            assert_within(compare(g, ref, "bf16"), "bf16")
            check_blocks(g["d_packed"], ref["d_packed"], "bf16")


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("N,BH", [(50, 400), (100, 333), (200, 301)])
def test_persistent_many_small_items(N, BH, d):
    """More work items than SMs, each with one to four 64-query sub-tiles: every
    persistent CTA walks several items whose first sub-tiles fall on either
    issuer's parity (one-sub-tile items leave an issuer without work in them),
    through the per-item K/V, accumulator-zeroing and epilogue barriers.  The
    fused mode on the GPU, every 64-query block of dQ and every 128-key block
    of dK/dV of sampled slices (the first, the last and ones in between)
    against the oracle."""
    inp = make_custom(BH=BH, N=N, d=d, dtype="bf16", seed=7000 + N + d)
    slices = sorted({0, 1, 2, 151, 152, 153, BH // 2, BH - 2, BH - 1})
    ref = oracle_fwd_bwd(inp, slices)
    g = gpu_fwd_bwd(inp, B.PSA_ALGO_TC)
    assert_within(compare(g, ref, "bf16", slices), "bf16")
    check_blocks(g["d_packed"], ref["d_packed"], "bf16", slices)


@pytest.mark.parametrize("d", [32, 64])
def test_timed_launches_match_oracle(d):
    """With kernel timing on, the tensor-core backward launches its kernels
    one after another (no programmatic dependent launch), with events around
    each; the results stay those of the oracle, and the timing records one
    launch of each backward kernel per call."""
    inp = make_custom(BH=20, N=1000, d=d, dtype="bf16", seed=900 + d)
    slices = [0, 19]
    ref = oracle_fwd_bwd(inp, slices)
    B.psa_attn_profile_read()
    B.psa_attn_profile_enable(True)
    try:
        gpu = gpu_fwd_bwd(inp, B.PSA_ALGO_TC)
    finally:
        B.psa_attn_profile_enable(False)
    prof = B.psa_attn_profile_read()
    errs = compare(gpu, ref, "bf16", slices)
    assert_within(errs, "bf16")
    check_blocks(gpu["d_packed"], ref["d_packed"], "bf16", slices)
    for slot in ("bwd_pre", "bwd_main", "bwd_dq"):
        ms, n = prof[slot]
        assert n >= 1 and ms > 0.0, (slot, prof)


@pytest.mark.parametrize("d", [16, 32, 64])
def test_fused_item_transitions_repeated(d):
    """The persistent fused kernel with several work items per CTA (64 slices
    of N = 1000: 512 units, ~3.4 per CTA, the last wave split), run five
    times: the first run matches the oracle on sampled slices, block by
    block, and every run agrees with it on every slice to rounding (the two
    MMA issuers' products of neighbouring sub-tiles, and the dQ reduces, may
    be summed in a different order), so a race between the item-crossing
    rings, K/V buffers or barriers in any slice would show."""
    inp = make_custom(BH=64, N=1000, d=d, dtype="bf16", seed=1100 + d)
    slices = [0, 31, 63]
    ref = oracle_fwd_bwd(inp, slices)
    first = gpu_fwd_bwd(inp, B.PSA_ALGO_TC)
    assert_within(compare(first, ref, "bf16", slices), "bf16")
    check_blocks(first["d_packed"], ref["d_packed"], "bf16", slices)
    runs = [first["d_packed"]] + [gpu_fwd_bwd(inp, B.PSA_ALGO_TC)["d_packed"] for _ in range(4)]
    for r in runs[1:]:
        for sec in range(4):
            assert rel_err(r[:, sec], runs[0][:, sec]) < 1e-2, sec
            for k0 in range(0, 1000, 128):
                blk = slice(k0, min(1000, k0 + 128))
                assert rel_err(r[:, sec, blk], runs[0][:, sec, blk]) < 2e-2, (sec, k0)
