"""Strided layouts (psa_attn_bwd_ex) and the merge op's backward
(psa_merge_bwd, psa_merge_attn_bwd): argument checks on the CPU (every error is
returned before anything is launched) and, on the GPU, parity with the fp64
oracle for padded rows, channel-major dO and dO read straight out of a merged
[B, c, H, W] gradient."""
import numpy as np
import pytest

from self_attention_backward_gb300 import binding as B
from self_attention_backward_gb300.inputs import make_custom

FAKE = 0x10000


@pytest.fixture(scope="module")
def lib():
    from self_attention_backward_gb300.build import build
    build()
    return B.lib()


def _ex(do_lo=None, do_hi=None, ldq=32, ldo=32, d=32, N=64, dtype=B.PSA_BF16, algo=B.PSA_ALGO_AUTO,
        ws_bytes=1 << 30, heads=2, Bn=1):
    row = B.psa_attn_view(FAKE, heads * N * d, N * d, d, 1)
    lo = do_lo if do_lo is not None else row
    hi = do_hi if do_hi is not None else row
    return B.psa_attn_bwd_ex(FAKE, ldq, FAKE, FAKE, ldo, FAKE, lo, hi, FAKE, FAKE, ws_bytes, Bn, heads, N, d, 0.1,
                             dtype, algo=algo, stream=0, check=False)


def test_ex_argument_errors(lib):
    cm = B.psa_attn_view(FAKE, 2 * 32 * 64, 32 * 64, 1, 64)          # channel-major [d, N]
    assert _ex(do_lo=B.psa_attn_view(0, 0, 0, 32, 1)) == B.PSA_ERR_ARG          # NULL base
    assert _ex(do_lo=B.psa_attn_view(FAKE + 2, 4096, 2048, 32, 1)) == B.PSA_ERR_ALIGN
    assert _ex(do_lo=B.psa_attn_view(FAKE, 4096, 2048, 2, 3)) == B.PSA_ERR_UNSUPPORTED   # neither layout
    assert _ex(do_lo=B.psa_attn_view(FAKE, 4096, 2048, 20, 1)) == B.PSA_ERR_UNSUPPORTED  # pos_stride < d
    assert _ex(do_lo=B.psa_attn_view(FAKE, -1, 2048, 32, 1)) == B.PSA_ERR_ARG
    # the tensor-core path needs 16-byte strides: a channel-major view with N = 100 (200-byte rows)
    cm100 = B.psa_attn_view(FAKE, 2 * 32 * 100, 32 * 100, 1, 100)
    assert _ex(do_lo=cm100, do_hi=cm100, N=100) == B.PSA_ERR_ALIGN
    assert _ex(do_lo=cm) == B.PSA_ERR_UNSUPPORTED                                # lo channel-major, hi rows
    assert _ex(ldq=16) == B.PSA_ERR_ARG                                           # row stride < d
    assert _ex(ldq=36) == B.PSA_ERR_ALIGN                                         # 72-byte rows
    assert _ex(ldq=40, algo=B.PSA_ALGO_SIMT) == B.PSA_ERR_UNSUPPORTED             # CUDA cores: plain rows
    assert _ex(algo=B.PSA_ALGO_TC_2PASS) == B.PSA_ERR_UNSUPPORTED
    assert _ex(dtype=B.PSA_F32, algo=B.PSA_ALGO_TC) == B.PSA_ERR_UNSUPPORTED
    assert _ex(ws_bytes=16) == B.PSA_ERR_WORKSPACE
    assert _ex(N=0) == B.PSA_OK                                                   # empty: nothing to do
    assert "16 bytes" in B.psa_attn_last_error() or B.psa_attn_last_error() == ""


def test_ex_workspace_sizes(lib):
    row = B.psa_attn_view(FAKE, 2 * 64 * 32, 64 * 32, 32, 1)
    cm = B.psa_attn_view(FAKE, 2 * 32 * 64, 32 * 64, 1, 64)
    plain = B.psa_attn_bwd_workspace_bytes(1, 2, 64, 32, B.PSA_F32, B.PSA_ALGO_SIMT)
    assert B.psa_attn_bwd_ex_workspace_bytes(row, row, 1, 2, 64, 32, B.PSA_F32, B.PSA_ALGO_SIMT) >= plain
    # the CUDA-core path gathers channel-major dO into the workspace: two more [BH, N, d] fp32 tensors
    gathered = B.psa_attn_bwd_ex_workspace_bytes(cm, cm, 1, 2, 64, 32, B.PSA_F32, B.PSA_ALGO_SIMT)
    assert gathered >= plain + 2 * 2 * 64 * 32 * 4
    assert B.psa_merge_attn_bwd_workspace_bytes(1, 2, 8, 8, 32, B.PSA_F32, B.PSA_ALGO_SIMT) == gathered
    assert B.psa_merge_attn_bwd_workspace_bytes(1, 2, 8, 8, 48, B.PSA_BF16, B.PSA_ALGO_AUTO) == 0


def test_merge_argument_errors(lib):
    assert B.psa_merge_bwd(FAKE, FAKE, FAKE, 1, 2, 4, 4, 32, 7, stream=0, check=False) == B.PSA_ERR_ARG
    assert B.psa_merge_bwd(None, FAKE, FAKE, 1, 2, 4, 4, 32, B.PSA_BF16, stream=0, check=False) == B.PSA_ERR_ARG
    assert B.psa_merge_bwd(FAKE, FAKE, FAKE, 1, 2, 4, 4, 256, B.PSA_BF16, stream=0, check=False) == \
        B.PSA_ERR_UNSUPPORTED
    assert B.psa_merge_bwd(FAKE, FAKE, FAKE, 0, 2, 4, 4, 32, B.PSA_BF16, stream=0, check=False) == B.PSA_OK
    # fused on the tensor cores: H*W = 9 positions make 18-byte rows of d_merged
    assert B.psa_merge_attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, 1, 2, 3, 3, 32, 0.1,
                                B.PSA_BF16, algo=B.PSA_ALGO_TC, stream=0, check=False) == B.PSA_ERR_ALIGN
    assert B.psa_merge_attn_bwd(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 1 << 30, 1, 2, 4, 4, 32, 0.1,
                                B.PSA_BF16, stream=0, check=False) == B.PSA_ERR_ARG


# ---------------------------------------------------------------- GPU parity
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _ref(inp, do_lo, do_hi):
    """fp64 oracle on the given (storage-rounded) inputs: d_packed [BH, 4, N, d]."""
    import oracle
    p = inp.packed.astype(np.float64)
    vs = np.ascontiguousarray(p[:, 2:4].transpose(1, 0, 2, 3))
    dq, dk, dvs = oracle.attn_bwd(p[:, 0], p[:, 1], vs, np.stack([do_lo, do_hi]).astype(np.float64), inp.scale)
    return np.stack([dq, dk, dvs[0], dvs[1]], axis=1)


def _check(got, ref, tol):
    from gpu_helpers import rel_err
    for s in range(4):
        e = rel_err(got[:, s], ref[:, s])
        assert e <= tol, (s, e)


@pytest.mark.gpu
@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("channel_major", [False, True])
def test_padded_rows_and_strided_do(lib, d, channel_major):
    """packed / d_packed rows padded to d + 8, O rows to d + 16, dO as a slice of a
    larger row-major or channel-major tensor with its own batch and head strides;
    the fused tensor-core path against the oracle, the padding left untouched."""
    torch = _gpu()
    from gpu_helpers import to_device
    Bn, heads, N = 2, 3, 200
    BH = Bn * heads
    inp = make_custom(BH=BH, N=N, d=d, dtype="bf16", seed=4100 + d + 7 * channel_major)
    dev = lambda a: to_device(a, "bf16")  # noqa: E731
    packed = dev(inp.packed)
    o_lo, o_hi, lse = B.attn_fwd(packed, inp.scale)
    packed_pad = torch.zeros((BH, 4, N, d + 8), dtype=torch.bfloat16, device="cuda")
    packed_pad[..., :d] = packed
    o_pad = [torch.zeros((BH, N, d + 16), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    o_pad[0][..., :d] = o_lo
    o_pad[1][..., :d] = o_hi
    views = []
    for g in (inp.do_lo, inp.do_hi):
        g4 = dev(g).reshape(Bn, heads, N, d)
        if channel_major:
            big = torch.zeros((Bn, heads + 1, d, N + 8), dtype=torch.bfloat16, device="cuda")
            big[:, :heads, :, :N] = g4.transpose(-1, -2)
            views.append(big[:, :heads, :, :N].transpose(-1, -2))
        else:
            big = torch.zeros((Bn + 1, heads, N + 3, d + 24), dtype=torch.bfloat16, device="cuda")
            big[:Bn, :, :N, :d] = g4
            views.append(big[:Bn, :, :N, :d])
    out = torch.full((BH, 4, N, d + 8), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.attn_bwd_ex(packed_pad, d, o_pad[0], o_pad[1], lse, views[0], views[1], inp.scale, heads, d_packed=out,
                  algo=B.PSA_ALGO_TC)
    B.psa_attn_sync_status()
    got = out.double().cpu().numpy()
    assert np.isnan(got[..., d:]).all()
    _check(got[..., :d], _ref(inp, inp.do_lo, inp.do_hi), 2e-2)


@pytest.mark.gpu
@pytest.mark.parametrize("d,H,W,dtype", [(32, 10, 12, "bf16"), (64, 20, 20, "bf16"), (16, 8, 8, "bf16"),
                                         (16, 4, 5, "f32")])
def test_merge_fused_matches_oracle(lib, d, H, W, dtype):
    """psa_merge_attn_bwd reads dO_lo / dO_hi straight out of d_merged [B, c, H, W];
    against the oracle's merge backward followed by its attention backward.  The
    plain psa_merge_bwd gather matches the oracle's merge backward bit for bit."""
    torch = _gpu()
    import oracle
    from gpu_helpers import to_device, TOL
    Bn, heads, N = 2, 2, H * W
    inp = make_custom(BH=Bn * heads, N=N, d=d, dtype=dtype, seed=4200 + d + H)
    rng = np.random.default_rng(4300 + d)
    from self_attention_backward_gb300.inputs import round_storage
    g = round_storage(rng.normal(size=(Bn, 2 * heads * d, H, W)), dtype)
    d_lo, d_hi = oracle.merge_bwd(g.reshape(Bn, 2 * heads * d, N).astype(np.float64), heads, d)
    packed = to_device(inp.packed, dtype)
    o_lo, o_hi, lse = B.attn_fwd(packed, inp.scale)
    gm = to_device(g, dtype)
    got = B.merge_attn_bwd(packed, o_lo, o_hi, lse, gm, heads, inp.scale)
    lo, hi = B.merge_bwd(gm, heads, d)
    B.psa_attn_sync_status()
    np.testing.assert_array_equal(lo.double().cpu().numpy(), d_lo)
    np.testing.assert_array_equal(hi.double().cpu().numpy(), d_hi)
    _check(got.double().cpu().numpy(), _ref(inp, d_lo, d_hi), TOL[dtype])
