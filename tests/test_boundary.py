"""The C-ABI library: it loads, exports every function include/psa_attn.h
declares, and rejects bad arguments before launching anything (no GPU needed:
every call below fails argument checks, so no CUDA call is made)."""

import pytest

from self_attention_backward_gb300 import binding as B


@pytest.fixture(scope="module")
def lib():
    try:
        from self_attention_backward_gb300.build import build
        build()
    except Exception as e:  # nvcc missing is a hard failure for this repo
        pytest.fail(f"CUDA library failed to build: {e}")
    return B.lib()


def test_exports_every_header_function(lib):
    names = B.header_functions()
    assert {"psa_attn_fwd", "psa_attn_bwd", "psa_attn_bwd_workspace_bytes", "psa_attn_last_error"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
        assert n in B._SIGS, f"binding lacks a signature for {n}"


def test_version(lib):
    assert B.psa_attn_version() >= 100


FAKE = 0x10000  # 16-byte aligned, never dereferenced: the calls fail checks first


def _fwd(**kw):
    a = dict(packed=FAKE, o_lo=FAKE, o_hi=FAKE, lse=FAKE, B=1, heads=2, N=16, head_dim=16, scale=0.25,
             dtype=B.PSA_F32, stream=0, check=False)
    a.update(kw)
    return B.psa_attn_fwd(**a)


def _bwd(**kw):
    a = dict(packed=FAKE, o_lo=FAKE, o_hi=FAKE, lse=FAKE, do_lo=FAKE, do_hi=FAKE, d_packed=FAKE,
             workspace=FAKE, workspace_bytes=0, B=1, heads=2, N=16, head_dim=16, scale=0.25,
             dtype=B.PSA_F32, stream=0, check=False)
    a.update(kw)
    return B.psa_attn_bwd(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=48), B.PSA_ERR_UNSUPPORTED),
    (dict(head_dim=128), B.PSA_ERR_UNSUPPORTED),
    (dict(N=-1), B.PSA_ERR_ARG),
    (dict(B=-2), B.PSA_ERR_ARG),
    (dict(dtype=7), B.PSA_ERR_ARG),
    (dict(scale=float("nan")), B.PSA_ERR_ARG),
    (dict(scale=float("inf")), B.PSA_ERR_ARG),
    (dict(packed=None), B.PSA_ERR_ARG),
    (dict(lse=None), B.PSA_ERR_ARG),
    (dict(o_hi=FAKE + 4), B.PSA_ERR_ALIGN),
    (dict(B=1 << 20, heads=1 << 10, N=1 << 12), B.PSA_ERR_UNSUPPORTED),
])
def test_fwd_rejects(lib, kw, code):
    assert _fwd(**kw) == code
    assert B.psa_attn_last_error() != ""


def test_fwd_empty_is_ok(lib):
    assert _fwd(N=0, packed=None, o_lo=None, o_hi=None, lse=None) == B.PSA_OK
    assert _fwd(B=0) == B.PSA_OK
    assert B.psa_attn_last_error() == ""


@pytest.mark.parametrize("kw,code", [
    (dict(d_packed=None), B.PSA_ERR_ARG),
    (dict(do_hi=FAKE + 8), B.PSA_ERR_ALIGN),
    (dict(workspace_bytes=0), B.PSA_ERR_WORKSPACE),
    (dict(workspace=None, workspace_bytes=1 << 20), B.PSA_ERR_WORKSPACE),
    (dict(workspace=FAKE + 2, workspace_bytes=1 << 20), B.PSA_ERR_ALIGN),
    (dict(head_dim=8), B.PSA_ERR_UNSUPPORTED),
])
def test_bwd_rejects(lib, kw, code):
    assert _bwd(**kw) == code


@pytest.mark.parametrize("algo", [B.PSA_ALGO_AUTO, B.PSA_ALGO_SIMT, B.PSA_ALGO_TC, B.PSA_ALGO_TC_2PASS])
@pytest.mark.parametrize("dtype", [B.PSA_F32, B.PSA_BF16])
def test_bwd_empty_is_ok(lib, algo, dtype):
    """An empty problem (N = 0 or B*heads = 0) returns PSA_OK without looking
    at any pointer or launching anything, for every kernel family that
    supports the dtype; the workspace it needs is 0 bytes."""
    tc = algo in (B.PSA_ALGO_TC, B.PSA_ALGO_TC_2PASS)
    want = B.PSA_ERR_UNSUPPORTED if (tc and dtype == B.PSA_F32) else B.PSA_OK
    none = dict(packed=None, o_lo=None, o_hi=None, lse=None, do_lo=None, do_hi=None, d_packed=None, workspace=None)
    assert _bwd(N=0, dtype=dtype, head_dim=32, algo=algo, **none) == want
    assert _bwd(B=0, dtype=dtype, head_dim=32, algo=algo, **none) == want
    assert B.psa_attn_bwd_workspace_bytes(1, 2, 0, 32, dtype, algo) == 0


def test_bwd_bad_algo(lib):
    assert _bwd(algo=9, workspace_bytes=1 << 20) == B.PSA_ERR_ARG


def test_bwd_tc_unsupported_for_fp32(lib):
    assert _bwd(algo=B.PSA_ALGO_TC, dtype=B.PSA_F32, workspace_bytes=1 << 20) == B.PSA_ERR_UNSUPPORTED
    assert _bwd(algo=B.PSA_ALGO_TC_2PASS, dtype=B.PSA_F32, workspace_bytes=1 << 20) == B.PSA_ERR_UNSUPPORTED
    assert _bwd(algo=B.PSA_ALGO_TC_2PASS + 1, workspace_bytes=1 << 20) == B.PSA_ERR_ARG


def test_two_pass_workspace_and_forward_rejects_it(lib):
    # the two-pass backward keeps only D (fp32 per query row, 256-byte aligned)
    assert B.psa_attn_bwd_workspace_bytes(2, 3, 100, 32, B.PSA_BF16, B.PSA_ALGO_TC_2PASS) == 2560
    assert B.psa_attn_bwd_workspace_bytes(1, 1, 100, 32, B.PSA_BF16, B.PSA_ALGO_TC_2PASS) == 512
    assert B.psa_attn_bwd_workspace_bytes(1, 1, 100, 32, B.PSA_F32, B.PSA_ALGO_TC_2PASS) == 0
    # the fused mode holds 8 bytes of statistics per query, padded to whole
    # 64-query sub-tiles, and an fp32 dQ accumulator
    assert B.psa_attn_bwd_workspace_bytes(1, 1, 100, 32, B.PSA_BF16, B.PSA_ALGO_TC) == 128 * 8 + 100 * 32 * 4
    rc = B.lib().psa_attn_fwd_algo(FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 16, 1.0, B.PSA_BF16, B.PSA_ALGO_TC_2PASS, None)
    assert rc == B.PSA_ERR_ARG


def test_workspace_bytes(lib):
    assert B.psa_attn_bwd_workspace_bytes(1, 2, 16, 16, B.PSA_F32) >= 2 * 16 * 4
    assert B.psa_attn_bwd_workspace_bytes(0, 2, 16, 16, B.PSA_F32) == 0
    assert B.psa_attn_bwd_workspace_bytes(1, 2, 16, 48, B.PSA_F32) == 0
    assert B.psa_attn_bwd_workspace_bytes(1, 2, 16, 16, B.PSA_F32, B.PSA_ALGO_SIMT) == 2 * 16 * 4
    # the check does not clobber the thread's last error
    _fwd(head_dim=48)
    msg = B.psa_attn_last_error()
    B.psa_attn_bwd_workspace_bytes(1, 2, 16, 48, B.PSA_F32)
    assert B.psa_attn_last_error() == msg


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        B.lib()


def _bwd_host(**kw):
    a = dict(packed=FAKE, o_lo=FAKE, o_hi=FAKE, lse=FAKE, do_lo=FAKE, do_hi=FAKE, d_packed=FAKE,
             dev_buf=FAKE * 16, dev_buf_bytes=0, B=1, heads=2, N=16, head_dim=16, scale=0.25,
             dtype=B.PSA_F32, algo=B.PSA_ALGO_AUTO, chunks=0, stream=0, check=False)
    a.update(kw)
    return B.psa_attn_bwd_host(**a)


def test_bwd_host_buffer_layout(lib):
    """The host entry point's device buffer: packed, o_lo, o_hi, do_lo, do_hi,
    lse, d_packed, then the workspace, each start 256-byte aligned."""
    a = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for (BH, N, d, dt, algo) in [(1, 100, 32, B.PSA_BF16, B.PSA_ALGO_TC), (3, 17, 16, B.PSA_F32, B.PSA_ALGO_AUTO),
                                 (2, 130, 64, B.PSA_BF16, B.PSA_ALGO_TC_2PASS)]:
        es = 2 if dt == B.PSA_BF16 else 4
        sec = BH * N * d * es
        ws = B.psa_attn_bwd_workspace_bytes(BH, 1, N, d, dt, algo)
        want = a(4 * sec) + 4 * a(sec) + a(BH * N * 4) + a(4 * sec) + a(ws)
        assert B.psa_attn_bwd_host_buffer_bytes(BH, 1, N, d, dt, algo) == want
    assert B.psa_attn_bwd_host_buffer_bytes(1, 1, 0, 32, B.PSA_BF16, B.PSA_ALGO_TC) == 0
    assert B.psa_attn_bwd_host_buffer_bytes(1, 1, 64, 48, B.PSA_BF16, B.PSA_ALGO_TC) == 0
    assert B.psa_attn_bwd_host_buffer_bytes(1, 1, 64, 32, B.PSA_F32, B.PSA_ALGO_TC) == 0
    assert B.psa_attn_bwd_host_buffer_bytes(1, 1, 64, 32, B.PSA_F32, 9) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(dev_buf_bytes=1), B.PSA_ERR_WORKSPACE),
    (dict(dev_buf=None, dev_buf_bytes=1 << 30), B.PSA_ERR_WORKSPACE),
    (dict(dev_buf=FAKE * 16 + 16, dev_buf_bytes=1 << 30), B.PSA_ERR_ALIGN),
    (dict(chunks=-1, dev_buf_bytes=1 << 30), B.PSA_ERR_ARG),
    (dict(chunks=65, dev_buf_bytes=1 << 30), B.PSA_ERR_ARG),
    (dict(packed=None, dev_buf_bytes=1 << 30), B.PSA_ERR_ARG),
    (dict(d_packed=None, dev_buf_bytes=1 << 30), B.PSA_ERR_ARG),
    (dict(scale=float("nan"), dev_buf_bytes=1 << 30), B.PSA_ERR_ARG),
    (dict(head_dim=48, dev_buf_bytes=1 << 30), B.PSA_ERR_UNSUPPORTED),
    (dict(N=-1), B.PSA_ERR_ARG),
    (dict(dtype=7), B.PSA_ERR_ARG),
    (dict(algo=9, dev_buf_bytes=1 << 30), B.PSA_ERR_ARG),
    (dict(algo=B.PSA_ALGO_TC, dev_buf_bytes=1 << 30), B.PSA_ERR_UNSUPPORTED),
    (dict(N=0, packed=None, dev_buf=None), B.PSA_OK),
    (dict(B=0, d_packed=None, dev_buf=None), B.PSA_OK),
])
def test_bwd_host_rejects_before_any_copy(lib, kw, code):
    """psa_attn_bwd_host checks sizes, dtype, algo, chunks, host pointers and
    its device buffer before it enqueues a copy (no GPU is touched here)."""
    assert _bwd_host(**kw) == code
    if code != B.PSA_OK:
        assert B.psa_attn_last_error()
