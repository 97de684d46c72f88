"""Pins for the fp64 CPU oracle (no GPU).

The pages print no worked example, so the oracle is pinned to mathematics that
does not go through its own code: central finite differences of its forward,
closed forms (N = 1, Q = 0, a two-key case written with the logistic function),
the float64 torch SDPA forward/autograd as an independent library routine, and
invariants of the softmax-attention gradient.  "Struct PsaFa2Backward"
(description, "Atomicity" paragraph) fixes that lo and hi share Q and K, that dQ
and dK are summed over the two calls and that each call owns its dV.
"""
import math

import numpy as np
import pytest

from self_attention_backward_gb300.inputs import make_inputs, make_custom

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _split(inp):
    p = inp.packed.astype(np.float64)
    q, k = p[:, 0], p[:, 1]
    vs = np.ascontiguousarray(p[:, 2:4].transpose(1, 0, 2, 3))
    dos = np.stack([inp.do_lo, inp.do_hi]).astype(np.float64)
    return q, k, vs, dos


def _loss(oracle_mod, q, k, vs, dos, scale):
    o, _ = oracle_mod.attn_fwd(q, k, vs, scale)
    return float(np.sum(o * dos))


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def _fd_grads(oracle_mod, q, k, vs, dos, scale, h=1e-5):
    """Central differences of L = sum_h <dO_h, O_h> w.r.t. every input element."""
    out = []
    for arr in (q, k, vs):
        g = np.zeros_like(arr)
        flat, gflat = arr.reshape(-1), g.reshape(-1)
        for idx in range(flat.size):
            old = flat[idx]
            flat[idx] = old + h
            lp = _loss(oracle_mod, q, k, vs, dos, scale)
            flat[idx] = old - h
            lm = _loss(oracle_mod, q, k, vs, dos, scale)
            flat[idx] = old
            gflat[idx] = (lp - lm) / (2 * h)
        out.append(g)
    return out


def test_fd_tiny_workload(oracle_mod):
    """Every input element of the 2-slice, N=16, d=16 fp32 workload."""
    inp = make_inputs("psa_f32_b1_h2_n16_d16")
    q, k, vs, dos = _split(inp)
    dq, dk, dvs = oracle_mod.attn_bwd(q, k, vs, dos, inp.scale)
    fq, fk, fv = _fd_grads(oracle_mod, q.copy(), k.copy(), vs.copy(), dos, inp.scale)
    assert _rel(dq, fq) < 1e-7
    assert _rel(dk, fk) < 1e-7
    assert _rel(dvs, fv) < 1e-7


@pytest.mark.parametrize("N", [1, 2, 3, 5])
@pytest.mark.parametrize("d", [1, 4])
@pytest.mark.parametrize("nv", [1, 2])
def test_fd_small(oracle_mod, N, d, nv):
    rng = np.random.default_rng(100 + 10 * N + d + nv)
    q, k = rng.normal(size=(2, 1, N, d))
    vs = rng.normal(size=(nv, 1, N, d))
    dos = rng.normal(size=(nv, 1, N, d))
    scale = 0.7
    dq, dk, dvs = oracle_mod.attn_bwd(q, k, vs, dos, scale)
    fq, fk, fv = _fd_grads(oracle_mod, q.copy(), k.copy(), vs.copy(), dos, scale)
    tol = 1e-7 * max(1.0, np.max(np.abs(fv)))
    assert np.max(np.abs(dq - fq)) < tol
    assert np.max(np.abs(dk - fk)) < tol
    assert np.max(np.abs(dvs - fv)) < tol


def test_torch_sdpa_two_calls(oracle_mod):
    """Two float64 torch SDPA calls (lo, hi) sharing q and k, autograd summing
    their dq/dk contributions -- the pair of calls the page describes."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    inp = make_custom(BH=3, N=23, d=8, dtype="f32", seed=7, scale=0.41)
    q, k, vs, dos = _split(inp)
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = [torch.tensor(vs[h], requires_grad=True) for h in range(2)]
    outs = [F.scaled_dot_product_attention(tq, tk, tv[h], scale=inp.scale) for h in range(2)]
    loss = sum((outs[h] * torch.tensor(dos[h])).sum() for h in range(2))
    loss.backward()
    dq, dk, dvs, o, lse, _ = oracle_mod.attn_bwd(q, k, vs, dos, inp.scale, want_fwd=True)
    assert _rel(o[0], outs[0].detach().numpy()) < 1e-13
    assert _rel(o[1], outs[1].detach().numpy()) < 1e-13
    tl = torch.logsumexp(inp.scale * torch.tensor(q) @ torch.tensor(k).transpose(-1, -2), dim=-1)
    assert _rel(lse, tl.numpy()) < 1e-13
    assert _rel(dq, tq.grad.numpy()) < 1e-12
    assert _rel(dk, tk.grad.numpy()) < 1e-12
    assert _rel(dvs[0], tv[0].grad.numpy()) < 1e-12
    assert _rel(dvs[1], tv[1].grad.numpy()) < 1e-12


def test_closed_form_n1(oracle_mod):
    """N = 1: O = V, LSE = scale <q, k>, dV = dO, dQ = dK = 0."""
    rng = np.random.default_rng(3)
    q, k = rng.normal(size=(2, 4, 1, 16))
    vs, dos = rng.normal(size=(2, 2, 4, 1, 16))
    dq, dk, dvs, o, lse, _ = oracle_mod.attn_bwd(q, k, vs, dos, 0.3, want_fwd=True)
    np.testing.assert_allclose(o, vs, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, 0.3 * np.sum(q * k, axis=-1), rtol=1e-14)
    np.testing.assert_allclose(dvs, dos, rtol=0, atol=1e-15)
    assert np.max(np.abs(dq)) < 1e-15 and np.max(np.abs(dk)) < 1e-15


def test_closed_form_q_zero(oracle_mod):
    """Q = 0: uniform softmax.  O_i = mean V, LSE = log N, dK = 0,
    dV_j = mean_i dO_i, dQ_i = (scale/N) sum_j <dO_i, V_j - mean V> k_j."""
    rng = np.random.default_rng(4)
    BH, N, d, scale = 2, 9, 5, 0.8
    q = np.zeros((BH, N, d))
    k = rng.normal(size=(BH, N, d))
    vs, dos = rng.normal(size=(2, 2, BH, N, d))
    dq, dk, dvs, o, lse, _ = oracle_mod.attn_bwd(q, k, vs, dos, scale, want_fwd=True)
    vbar = vs.mean(axis=2, keepdims=True)                   # [2, BH, 1, d]
    np.testing.assert_allclose(o, np.broadcast_to(vbar, o.shape), atol=1e-14)
    np.testing.assert_allclose(lse, np.full((BH, N), math.log(N)), rtol=1e-14)
    assert np.max(np.abs(dk)) < 1e-14
    np.testing.assert_allclose(dvs, np.broadcast_to(dos.mean(axis=2, keepdims=True), dvs.shape), atol=1e-14)
    # c_ij = sum_h <dO_h[i], V_h[j] - Vbar_h>
    c = np.einsum("hbic,hbjc->bij", dos, vs - vbar)
    expect = scale / N * np.einsum("bij,bjc->bic", c, k)
    np.testing.assert_allclose(dq, expect, atol=1e-13)


def test_closed_form_two_keys(oracle_mod):
    """N = 2, d = 1, one V: row i's softmax is the logistic function of
    z_i = scale q_i (k_0 - k_1), so O_i = v_1 + sig(z_i) (v_0 - v_1) and every
    gradient follows from sig' = sig (1 - sig)."""
    q = np.array([[[0.9], [-1.7]]])
    k = np.array([[[0.4], [1.3]]])
    v = np.array([[[[2.0], [-0.5]]]])
    do = np.array([[[[0.3], [-1.1]]]])
    scale = 0.75
    dq, dk, dvs, o, lse, _ = oracle_mod.attn_bwd(q, k, v, do, scale, want_fwd=True)
    qi, k0, k1, v0, v1, g = q[0, :, 0], k[0, 0, 0], k[0, 1, 0], v[0, 0, 0, 0], v[0, 0, 1, 0], do[0, 0, :, 0]
    z = scale * qi * (k0 - k1)
    sig = 1.0 / (1.0 + np.exp(-z))
    dsig = sig * (1.0 - sig)
    np.testing.assert_allclose(o[0, 0, :, 0], v1 + sig * (v0 - v1), rtol=1e-14)
    np.testing.assert_allclose(lse[0], scale * qi * k1 + np.log1p(np.exp(z)), rtol=1e-14)
    np.testing.assert_allclose(dq[0, :, 0], g * (v0 - v1) * dsig * scale * (k0 - k1), rtol=1e-13)
    dk0 = np.sum(g * (v0 - v1) * dsig * scale * qi)
    np.testing.assert_allclose(dk[0, :, 0], [dk0, -dk0], rtol=1e-13)
    np.testing.assert_allclose(dvs[0, 0, :, 0], [np.sum(g * sig), np.sum(g * (1 - sig))], rtol=1e-14)


@pytest.fixture(scope="module")
def mid_case():
    inp = make_custom(BH=2, N=37, d=8, dtype="f32", seed=11, scale=0.5)
    return _split(inp) + (inp.scale,)


def test_equal_v_rows_zero_dqdk(oracle_mod, mid_case):
    """All rows of V_lo equal and all rows of V_hi equal: dP_ij = D_i, so dS = 0."""
    q, k, vs, dos, scale = mid_case
    vs = np.broadcast_to(vs[:, :, :1, :], vs.shape).copy()
    dq, dk, dvs = oracle_mod.attn_bwd(q, k, vs, dos, scale)
    assert np.max(np.abs(dq)) < 1e-13 and np.max(np.abs(dk)) < 1e-13
    assert np.max(np.abs(dvs)) > 0.1


def test_dv_column_sums(oracle_mod, mid_case):
    """Rows of P sum to 1, so sum_j dV_h[j] = sum_i dO_h[i]."""
    q, k, vs, dos, scale = mid_case
    _, _, dvs = oracle_mod.attn_bwd(q, k, vs, dos, scale)
    np.testing.assert_allclose(dvs.sum(axis=2), dos.sum(axis=2), atol=1e-12)


def test_dk_sums_to_zero_and_scaling_identity(oracle_mod, mid_case):
    """sum_j dS_ij = 0 gives sum_j dK_j = 0; S invariant under Q -> aQ, K -> K/a
    gives sum_i <q_i, dQ_i> = sum_j <k_j, dK_j>."""
    q, k, vs, dos, scale = mid_case
    dq, dk, _ = oracle_mod.attn_bwd(q, k, vs, dos, scale)
    assert np.max(np.abs(dk.sum(axis=1))) < 1e-12 * max(1.0, np.max(np.abs(dk)))
    np.testing.assert_allclose(np.sum(q * dq, axis=(1, 2)), np.sum(k * dk, axis=(1, 2)), rtol=1e-11)


def test_key_and_query_permutation(oracle_mod, mid_case):
    q, k, vs, dos, scale = mid_case
    dq, dk, dvs, o, _, _ = oracle_mod.attn_bwd(q, k, vs, dos, scale, want_fwd=True)
    perm = np.random.default_rng(5).permutation(q.shape[1])
    # permuting keys (K and V rows together) permutes dK, dV; dQ and O unchanged
    dq2, dk2, dvs2, o2, _, _ = oracle_mod.attn_bwd(q, k[:, perm], vs[:, :, perm], dos, scale, want_fwd=True)
    np.testing.assert_allclose(dq2, dq, atol=1e-13)
    np.testing.assert_allclose(o2, o, atol=1e-13)
    np.testing.assert_allclose(dk2, dk[:, perm], atol=1e-13)
    np.testing.assert_allclose(dvs2, dvs[:, :, perm], atol=1e-13)
    # permuting queries (Q and dO rows together) permutes dQ, O; dK, dV unchanged
    dq3, dk3, dvs3, o3, _, _ = oracle_mod.attn_bwd(q[:, perm], k, vs, dos[:, :, perm], scale, want_fwd=True)
    np.testing.assert_allclose(dq3, dq[:, perm], atol=1e-13)
    np.testing.assert_allclose(o3, o[:, :, perm], atol=1e-13)
    np.testing.assert_allclose(dk3, dk, atol=1e-13)
    np.testing.assert_allclose(dvs3, dvs, atol=1e-13)


def test_pair_is_sum_of_single_calls(oracle_mod, mid_case):
    """The lo/hi pair's dQ, dK equal the sums of two independent one-V backward
    passes, and each dV equals that call's own dV."""
    q, k, vs, dos, scale = mid_case
    dq, dk, dvs = oracle_mod.attn_bwd(q, k, vs, dos, scale)
    dq_lo, dk_lo, dv_lo = oracle_mod.attn_bwd(q, k, vs[:1], dos[:1], scale)
    dq_hi, dk_hi, dv_hi = oracle_mod.attn_bwd(q, k, vs[1:], dos[1:], scale)
    np.testing.assert_allclose(dq, dq_lo + dq_hi, atol=1e-13)
    np.testing.assert_allclose(dk, dk_lo + dk_hi, atol=1e-13)
    np.testing.assert_allclose(dvs[0], dv_lo[0], atol=1e-14)
    np.testing.assert_allclose(dvs[1], dv_hi[0], atol=1e-14)


def test_packed_wrappers(oracle_mod):
    inp = make_custom(BH=2, N=11, d=4, dtype="bf16", seed=2)
    dp = oracle_mod.psa_bwd(inp.packed, inp.do_lo, inp.do_hi, inp.scale)
    q, k, vs, dos = _split(inp)
    dq, dk, dvs = oracle_mod.attn_bwd(q, k, vs, dos, inp.scale)
    assert dp.shape == (2, 4, 11, 4)
    np.testing.assert_array_equal(dp[:, 0], dq)
    np.testing.assert_array_equal(dp[:, 1], dk)
    np.testing.assert_array_equal(dp[:, 2], dvs[0])
    np.testing.assert_array_equal(dp[:, 3], dvs[1])
    o_lo, o_hi, lse = oracle_mod.psa_fwd(inp.packed, inp.scale)
    assert o_lo.shape == (2, 11, 4) and lse.shape == (2, 11)


def test_empty_and_bad_sizes(oracle_mod):
    z = np.zeros((0, 4, 4))
    dq, dk, dvs = oracle_mod.attn_bwd(z, z, np.zeros((2, 0, 4, 4)), np.zeros((2, 0, 4, 4)), 1.0)
    assert dq.shape == (0, 4, 4) and dvs.shape == (2, 0, 4, 4)
    with pytest.raises(RuntimeError):
        oracle_mod.attn_fwd(np.zeros((1, 2, 0)), np.zeros((1, 2, 0)), np.zeros((1, 1, 2, 0)), 1.0)


def test_thread_count_independent(oracle_mod):
    """Rows are independent; the result must not depend on the thread count."""
    inp = make_custom(BH=2, N=40, d=8, dtype="f32", seed=9)
    q, k, vs, dos = _split(inp)
    n0 = oracle_mod.threads()
    try:
        oracle_mod.set_threads(1)
        a = oracle_mod.attn_bwd(q, k, vs, dos, inp.scale)
        oracle_mod.set_threads(max(2, n0))
        b = oracle_mod.attn_bwd(q, k, vs, dos, inp.scale)
    finally:
        oracle_mod.set_threads(n0)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


# ---------------------------------------------------------------- the merge op
def test_merge_bwd_index_map(oracle_mod):
    """The merge's backward against the reading written as a closed form of the
    indices: with d_merged[b, ch, n] = 1000 b + 10 ch + n, dO_lo[b*heads + h, n, j]
    must be 1000 b + 10 (h d + j) + n and dO_hi the same with ch shifted by heads d
    (lo channels first, head-major within each half)."""
    B, heads, d, N = 2, 3, 2, 5
    b, ch, n = np.meshgrid(np.arange(B), np.arange(2 * heads * d), np.arange(N), indexing="ij")
    g = 1000.0 * b + 10.0 * ch + n
    d_lo, d_hi = oracle_mod.merge_bwd(g, heads, d)
    for bb in range(B):
        for h in range(heads):
            for nn in range(N):
                for j in range(d):
                    assert d_lo[bb * heads + h, nn, j] == 1000 * bb + 10 * (h * d + j) + nn
                    assert d_hi[bb * heads + h, nn, j] == 1000 * bb + 10 * (heads * d + h * d + j) + nn


def test_merge_backward_is_the_adjoint_and_inverse(oracle_mod):
    """The merge is a permutation of elements: its backward is the adjoint of the
    forward (<M x, g> = <x, M^T g>) and inverts it."""
    rng = np.random.default_rng(7)
    B, heads, N, d = 2, 3, 7, 4
    o_lo, o_hi = rng.normal(size=(2, B * heads, N, d))
    g = rng.normal(size=(B, 2 * heads * d, N))
    m = oracle_mod.merge_fwd(o_lo, o_hi, B, heads)
    g_lo, g_hi = oracle_mod.merge_bwd(g, heads, d)
    assert abs(np.sum(m * g) - (np.sum(o_lo * g_lo) + np.sum(o_hi * g_hi))) < 1e-10
    r_lo, r_hi = oracle_mod.merge_bwd(m, heads, d)
    np.testing.assert_array_equal(r_lo, o_lo)
    np.testing.assert_array_equal(r_hi, o_hi)
    assert sorted(m.ravel()) == sorted(np.concatenate([o_lo.ravel(), o_hi.ravel()]))


def test_merged_backward_against_finite_differences(oracle_mod):
    """The attention backward fed by the merge's backward is the gradient of
    L = <merge(O_lo, O_hi), G> with respect to Q, K and V (central differences
    over every input element of a tiny case)."""
    rng = np.random.default_rng(11)
    B, heads, N, d = 1, 2, 3, 2
    q, k = rng.normal(size=(2, B * heads, N, d))
    vs = rng.normal(size=(2, B * heads, N, d))
    G = rng.normal(size=(B, 2 * heads * d, N))
    scale = 0.7

    def loss():
        o, _ = oracle_mod.attn_fwd(q, k, vs, scale)
        return float(np.sum(oracle_mod.merge_fwd(o[0], o[1], B, heads) * G))

    dos = np.stack(oracle_mod.merge_bwd(G, heads, d))
    dq, dk, dvs = oracle_mod.attn_bwd(q, k, vs, dos, scale)
    h = 1e-5
    for arr, grad in ((q, dq), (k, dk), (vs, dvs)):
        flat, gflat = arr.reshape(-1), grad.reshape(-1)
        for idx in range(flat.size):
            old = flat[idx]
            flat[idx] = old + h
            lp = loss()
            flat[idx] = old - h
            lm = loss()
            flat[idx] = old
            assert abs((lp - lm) / (2 * h) - gflat[idx]) < 1e-7 * max(1.0, abs(gflat[idx]))
