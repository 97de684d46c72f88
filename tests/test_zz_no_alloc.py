"""psa_attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (a plugin handed only its tensors by a host runtime that owns the
memory, or an application that forbids allocation after start-up).  Its
scratch is a static array inside the library, so it takes no workspace.

This file is collected last on purpose: the GPU test must pass both in a fresh
process and after every other test has run in the same process."""
import numpy as np
import pytest

from self_attention_backward_gb300 import binding as B
from self_attention_backward_gb300.inputs import make_custom

FAKE = 0x10000


def _lib():
    from self_attention_backward_gb300.build import build
    build()
    return B.lib()


def test_noalloc_rejects_oversize_before_launch():
    """Sizes over the static scratch are refused with a clear error (no GPU call)."""
    _lib()
    cap = B.psa_attn_bwd_noalloc_max_rows()
    assert cap == 1 << 19
    rc = B.psa_attn_bwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, cap + 1, 32, 0.1,
                                dtype=B.PSA_BF16, stream=0, check=False)
    assert rc == B.PSA_ERR_UNSUPPORTED
    assert "static scratch" in B.psa_attn_last_error()
    rc = B.psa_attn_bwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 1, 16, 32, 0.1,
                                dtype=B.PSA_BF16, stream=0, check=False)
    assert rc == B.PSA_ERR_ARG


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_two_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _lib()
    from gpu_helpers import TOL, oracle_fwd_bwd, rel_err, to_device

    # two calls in a row: a larger problem, then a smaller one that reuses the
    # same static scratch (stale rows from the first call must not leak in)
    cases = [make_custom(BH=6, N=700, d=32, dtype="bf16", seed=501),
             make_custom(BH=2, N=129, d=64, dtype="f32", seed=502)]
    for inp in cases:
        BH, _, N, d = inp.packed.shape
        packed = to_device(inp.packed, inp.dtype)
        do_lo, do_hi = to_device(inp.do_lo, inp.dtype), to_device(inp.do_hi, inp.dtype)
        o_lo, o_hi, lse = B.attn_fwd(packed, inp.scale)
        ref = B.attn_bwd(packed, o_lo, o_hi, lse, do_lo, do_hi, inp.scale)      # workspace entry point
        got = torch.full_like(packed, float("nan"))
        B.psa_attn_bwd_noalloc(packed, o_lo, o_hi, lse, do_lo, do_hi, got, BH, 1, N, d, inp.scale)
        B.psa_attn_sync_status()
        g, r = got.double().cpu().numpy(), ref.double().cpu().numpy()
        assert np.isfinite(g).all()
        oracle = oracle_fwd_bwd(inp)["d_packed"]
        for s in range(4):
            assert rel_err(g[:, s], r[:, s]) <= TOL[inp.dtype], (inp.dtype, s)
            # and against the fp64 oracle itself, not only the other entry point
            assert rel_err(g[:, s], oracle[:, s]) <= TOL[inp.dtype], (inp.dtype, s, "oracle")
