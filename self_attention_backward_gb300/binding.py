"""ctypes binding of the C ABI in ``include/psa_attn.h`` (argument marshalling only).

Every function here turns torch tensors into device pointers and sizes and
calls the C entry point of the same name; all arithmetic runs in the CUDA
library.  There is no fallback: if ``_psa_attn.so`` is missing, the first call
raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_psa_attn.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "psa_attn.h")

PSA_F32, PSA_BF16 = 0, 1
PSA_OK, PSA_ERR_ARG, PSA_ERR_ALIGN, PSA_ERR_UNSUPPORTED = 0, -1, -2, -3
PSA_ERR_WORKSPACE, PSA_ERR_CUDA, PSA_ERR_TIMEOUT = -4, -5, -6
PSA_ALGO_AUTO, PSA_ALGO_SIMT, PSA_ALGO_TC, PSA_ALGO_TC_2PASS = 0, 1, 2, 3

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_ll = ctypes.c_longlong


class psa_attn_view(ctypes.Structure):
    """A strided view of a [B, heads, N, d] tensor (strides in elements), as in
    include/psa_attn.h."""
    _fields_ = [("base", ctypes.c_void_p), ("batch_stride", ctypes.c_longlong), ("head_stride", ctypes.c_longlong),
                ("pos_stride", ctypes.c_longlong), ("feat_stride", ctypes.c_longlong)]


_vw = ctypes.POINTER(psa_attn_view)
_SIGS = {
    "psa_attn_fwd": ([_vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp], _i),
    "psa_attn_fwd_algo": ([_vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _vp], _i),
    "psa_attn_bwd_workspace_bytes": ([_i, _i, _i, _i, _i], _sz),
    "psa_attn_bwd_workspace_bytes_algo": ([_i, _i, _i, _i, _i, _i], _sz),
    "psa_attn_bwd": ([_vp] * 8 + [_sz, _i, _i, _i, _i, _f, _i, _vp], _i),
    "psa_attn_bwd_algo": ([_vp] * 8 + [_sz, _i, _i, _i, _i, _f, _i, _i, _vp], _i),
    "psa_attn_bwd_noalloc": ([_vp] * 7 + [_i, _i, _i, _i, _f, _i, _vp], _i),
    "psa_attn_bwd_noalloc_max_rows": ([], ctypes.c_longlong),
    "psa_attn_bwd_host": ([_vp] * 8 + [_sz, _i, _i, _i, _i, _f, _i, _i, _i, _vp], _i),
    "psa_attn_bwd_host_buffer_bytes": ([_i, _i, _i, _i, _i, _i], _sz),
    "psa_attn_bwd_host_chunks": ([_i, _i, _i, _i, _i, _i], _i),
    "psa_attn_sync_status": ([_vp], _i),
    "psa_attn_selftest_wait_timeout": ([_vp], _i),
    "psa_attn_profile_enable": ([_i], _i),
    "psa_attn_profile_read": ([ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int), _i], _i),
    "psa_attn_profile_slot_name": ([_i], ctypes.c_char_p),
    "psa_attn_last_error": ([], ctypes.c_char_p),
    "psa_attn_version": ([], _i),
    "psa_attn_bwd_ex": ([_vp, _ll, _vp, _vp, _ll, _vp, _vw, _vw, _vp, _vp, _sz, _i, _i, _i, _i, _f, _i, _i, _vp], _i),
    "psa_attn_bwd_ex_workspace_bytes": ([_vw, _vw, _i, _i, _i, _i, _i, _i], _sz),
    "psa_merge_bwd": ([_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp], _i),
    "psa_merge_attn_bwd": ([_vp] * 6 + [_vp, _sz, _i, _i, _i, _i, _i, _f, _i, _i, _vp], _i),
    "psa_merge_attn_bwd_workspace_bytes": ([_i] * 7, _sz),
}

_lock = threading.Lock()
_lib = None


class PsaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"psa status {code}: {msg}")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"CUDA library {LIB_PATH} is not built; run "
                                   "`python -m self_attention_backward_gb300.build` (nvcc, sm_103a)")
            L = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in _SIGS.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/psa_attn.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(psa_\w+)\s*\(", text)))


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return PSA_F32
    if t.dtype == torch.bfloat16:
        return PSA_BF16
    raise TypeError(f"unsupported storage dtype {t.dtype}")


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int) -> int:
    if rc != PSA_OK:
        raise PsaError(rc, psa_attn_last_error())
    return rc


def psa_attn_last_error() -> str:
    return lib().psa_attn_last_error().decode()


def psa_attn_version() -> int:
    return int(lib().psa_attn_version())


def psa_attn_fwd(packed, o_lo, o_hi, lse, B, heads, N, head_dim, scale, dtype=None, stream=None,
                 check=True, algo=PSA_ALGO_AUTO) -> int:
    dtype = _dtype_code(packed) if dtype is None else dtype
    rc = lib().psa_attn_fwd_algo(_ptr(packed), _ptr(o_lo), _ptr(o_hi), _ptr(lse), B, heads, N, head_dim,
                                 float(scale), dtype, algo, _stream(stream))
    return _check(rc) if check else rc


def psa_attn_bwd_workspace_bytes(B, heads, N, head_dim, dtype, algo=PSA_ALGO_AUTO) -> int:
    return int(lib().psa_attn_bwd_workspace_bytes_algo(B, heads, N, head_dim, dtype, algo))


def psa_attn_bwd(packed, o_lo, o_hi, lse, do_lo, do_hi, d_packed, workspace, workspace_bytes,
                 B, heads, N, head_dim, scale, dtype=None, stream=None, algo=PSA_ALGO_AUTO,
                 check=True) -> int:
    dtype = _dtype_code(packed) if dtype is None else dtype
    rc = lib().psa_attn_bwd_algo(_ptr(packed), _ptr(o_lo), _ptr(o_hi), _ptr(lse), _ptr(do_lo), _ptr(do_hi),
                                 _ptr(d_packed), _ptr(workspace), int(workspace_bytes), B, heads, N,
                                 head_dim, float(scale), dtype, algo, _stream(stream))
    return _check(rc) if check else rc


def psa_attn_bwd_noalloc(packed, o_lo, o_hi, lse, do_lo, do_hi, d_packed, B, heads, N, head_dim, scale,
                         dtype=None, stream=None, check=True) -> int:
    """Backward without a workspace argument: its scratch is a static array in
    the library (see include/psa_attn.h).  For callers that cannot allocate."""
    dtype = _dtype_code(packed) if dtype is None else dtype
    rc = lib().psa_attn_bwd_noalloc(_ptr(packed), _ptr(o_lo), _ptr(o_hi), _ptr(lse), _ptr(do_lo), _ptr(do_hi),
                                    _ptr(d_packed), B, heads, N, head_dim, float(scale), dtype, _stream(stream))
    return _check(rc) if check else rc


def psa_attn_bwd_noalloc_max_rows() -> int:
    return int(lib().psa_attn_bwd_noalloc_max_rows())


def psa_attn_bwd_host(packed, o_lo, o_hi, lse, do_lo, do_hi, d_packed, dev_buf, dev_buf_bytes,
                      B, heads, N, head_dim, scale, dtype=None, algo=PSA_ALGO_AUTO, chunks=0, stream=None,
                      check=True) -> int:
    """Backward on HOST tensors (ideally pinned), `dev_buf` a device scratch of
    psa_attn_bwd_host_buffer_bytes(...) bytes (see include/psa_attn.h)."""
    dtype = _dtype_code(packed) if dtype is None else dtype
    rc = lib().psa_attn_bwd_host(_ptr(packed), _ptr(o_lo), _ptr(o_hi), _ptr(lse), _ptr(do_lo), _ptr(do_hi),
                                 _ptr(d_packed), _ptr(dev_buf), int(dev_buf_bytes), B, heads, N, head_dim,
                                 float(scale), dtype, algo, int(chunks), _stream(stream))
    return _check(rc) if check else rc


def psa_attn_bwd_host_buffer_bytes(B, heads, N, head_dim, dtype, algo=PSA_ALGO_AUTO) -> int:
    return int(lib().psa_attn_bwd_host_buffer_bytes(B, heads, N, head_dim, dtype, algo))


def psa_attn_bwd_host_chunks(B, heads, N, head_dim, dtype, algo=PSA_ALGO_AUTO) -> int:
    return int(lib().psa_attn_bwd_host_chunks(B, heads, N, head_dim, dtype, algo))


def psa_attn_sync_status(stream=None, check=True) -> int:
    rc = lib().psa_attn_sync_status(_stream(stream))
    return _check(rc) if check else rc


def psa_attn_selftest_wait_timeout(stream=None, check=True) -> int:
    rc = lib().psa_attn_selftest_wait_timeout(_stream(stream))
    return _check(rc) if check else rc


def psa_attn_profile_enable(on: bool = True) -> int:
    return _check(lib().psa_attn_profile_enable(1 if on else 0))


def psa_attn_profile_slot_name(slot: int) -> str:
    return lib().psa_attn_profile_slot_name(slot).decode()


def psa_attn_profile_read() -> dict:
    """{slot name: (total ms, launches)} since the last read; clears the records."""
    n = 4
    ms = (ctypes.c_float * n)()
    cnt = (ctypes.c_int * n)()
    rc = lib().psa_attn_profile_read(ms, cnt, n)
    if rc < 0:
        raise PsaError(rc, psa_attn_last_error())
    return {psa_attn_profile_slot_name(i): (float(ms[i]), int(cnt[i])) for i in range(rc)}


# ----------------------------------------------------------------- helpers
def _torch_dtype(dtype):
    import torch
    return {PSA_F32: torch.float32, PSA_BF16: torch.bfloat16}[dtype]


def attn_fwd(packed, scale: float, stream=None, algo=PSA_ALGO_AUTO):
    """Allocates O_lo, O_hi, LSE on packed's device and runs psa_attn_fwd.

    packed: [BH, 4, N, d] CUDA tensor (fp32 or bf16).  B is taken as BH, heads 1.
    """
    import torch
    BH, four, N, d = packed.shape
    assert four == 4 and packed.is_contiguous()
    o_lo = torch.empty((BH, N, d), dtype=packed.dtype, device=packed.device)
    o_hi = torch.empty_like(o_lo)
    lse = torch.empty((BH, N), dtype=torch.float32, device=packed.device)
    psa_attn_fwd(packed, o_lo, o_hi, lse, BH, 1, N, d, scale, stream=stream, algo=algo)
    return o_lo, o_hi, lse


class BwdWorkspace:
    """A device workspace sized for psa_attn_bwd, grown on demand."""

    def __init__(self, device="cuda"):
        self.device = device
        self.buf = None

    def get(self, nbytes: int):
        import torch
        if nbytes == 0:
            return None
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        return self.buf


def attn_bwd(packed, o_lo, o_hi, lse, do_lo, do_hi, scale: float, d_packed=None, workspace=None,
             algo=PSA_ALGO_AUTO, stream=None):
    """Runs psa_attn_bwd; returns d_packed [BH, 4, N, d] (dQ, dK, dV_lo, dV_hi)."""
    import torch
    BH, _, N, d = packed.shape
    dt = _dtype_code(packed)
    if d_packed is None:
        d_packed = torch.empty_like(packed)
    nbytes = psa_attn_bwd_workspace_bytes(BH, 1, N, d, dt, algo)
    ws = (workspace or BwdWorkspace(packed.device)).get(nbytes)
    psa_attn_bwd(packed, o_lo, o_hi, lse, do_lo, do_hi, d_packed, ws, nbytes, BH, 1, N, d, scale,
                 dtype=dt, stream=stream, algo=algo)
    return d_packed


class HostBwd:
    """psa_attn_bwd_host for one shape: the device buffer it needs (the
    device copies of the inputs and of d_packed, and the workspace) is
    allocated once here, by torch; each call passes the host tensors (pinned
    for asynchronous copies) to the native entry point, which pipelines the
    copies in, the backward and the copy back over `chunks` groups of
    (batch*head) slices (None = the library's choice)."""

    def __init__(self, BH: int, N: int, d: int, dtype: int, device="cuda", algo=PSA_ALGO_AUTO, chunks=None):
        import torch
        self.shape = (BH, N, d)
        self.dtype, self.algo = dtype, algo
        self.chunks = 0 if chunks is None else int(chunks)
        self.buf_bytes = psa_attn_bwd_host_buffer_bytes(BH, 1, N, d, dtype, algo)
        self.buf = torch.empty(max(self.buf_bytes, 1), dtype=torch.uint8, device=device)
        es = 2 if dtype == PSA_BF16 else 4
        self._in_bytes = BH * N * (8 * d * es + 4)
        self._out_bytes = BH * N * 4 * d * es

    def h2d_bytes(self) -> int:
        return self._in_bytes

    def d2h_bytes(self) -> int:
        return self._out_bytes

    def __call__(self, packed, o_lo, o_hi, lse, do_lo, do_hi, scale: float, out, stream=None):
        BH, N, d = self.shape
        psa_attn_bwd_host(packed, o_lo, o_hi, lse, do_lo, do_hi, out, self.buf, self.buf_bytes, BH, 1, N, d,
                          scale, dtype=self.dtype, algo=self.algo, chunks=self.chunks, stream=stream)
        return out


# ----------------------------------------------------------------- strided layouts and the merge
def view_of(t) -> psa_attn_view:
    """psa_attn_view of a 4-D torch tensor [B, heads, N, d] with any strides."""
    assert t.dim() == 4
    sb, sh, sn, sj = t.stride()
    return psa_attn_view(t.data_ptr(), sb, sh, sn, sj)


def psa_attn_bwd_ex(packed, qkv_row_stride, o_lo, o_hi, o_row_stride, lse, do_lo: psa_attn_view,
                    do_hi: psa_attn_view, d_packed, workspace, workspace_bytes, B, heads, N, head_dim, scale,
                    dtype, algo=PSA_ALGO_AUTO, stream=None, check=True) -> int:
    rc = lib().psa_attn_bwd_ex(_ptr(packed), int(qkv_row_stride), _ptr(o_lo), _ptr(o_hi), int(o_row_stride),
                               _ptr(lse), ctypes.byref(do_lo), ctypes.byref(do_hi), _ptr(d_packed), _ptr(workspace),
                               int(workspace_bytes), B, heads, N, head_dim, float(scale), dtype, algo,
                               _stream(stream))
    return _check(rc) if check else rc


def psa_attn_bwd_ex_workspace_bytes(do_lo: psa_attn_view, do_hi: psa_attn_view, B, heads, N, head_dim, dtype,
                                    algo=PSA_ALGO_AUTO) -> int:
    return int(lib().psa_attn_bwd_ex_workspace_bytes(ctypes.byref(do_lo), ctypes.byref(do_hi), B, heads, N,
                                                     head_dim, dtype, algo))


def psa_merge_bwd(d_merged, d_lo, d_hi, B, heads, H, W, head_dim, dtype, stream=None, check=True) -> int:
    rc = lib().psa_merge_bwd(_ptr(d_merged), _ptr(d_lo), _ptr(d_hi), B, heads, H, W, head_dim, dtype,
                             _stream(stream))
    return _check(rc) if check else rc


def psa_merge_attn_bwd(packed, o_lo, o_hi, lse, d_merged, d_packed, workspace, workspace_bytes, B, heads, H, W,
                       head_dim, scale, dtype, algo=PSA_ALGO_AUTO, stream=None, check=True) -> int:
    rc = lib().psa_merge_attn_bwd(_ptr(packed), _ptr(o_lo), _ptr(o_hi), _ptr(lse), _ptr(d_merged), _ptr(d_packed),
                                  _ptr(workspace), int(workspace_bytes), B, heads, H, W, head_dim, float(scale),
                                  dtype, algo, _stream(stream))
    return _check(rc) if check else rc


def psa_merge_attn_bwd_workspace_bytes(B, heads, H, W, head_dim, dtype, algo=PSA_ALGO_AUTO) -> int:
    return int(lib().psa_merge_attn_bwd_workspace_bytes(B, heads, H, W, head_dim, dtype, algo))


def attn_bwd_ex(packed, d, o_lo, o_hi, lse, do_lo4, do_hi4, scale: float, heads: int, d_packed=None,
                workspace=None, algo=PSA_ALGO_AUTO, stream=None):
    """psa_attn_bwd_ex on torch tensors: packed [BH, 4, N, ld] (rows of d used),
    o_lo / o_hi [BH, N, ld_o], do_lo4 / do_hi4 any 4-D [B, heads, N, d] views
    (their torch strides are passed through).  Returns d_packed, shaped like
    packed (only the first d elements of each row are written)."""
    import torch
    BH, _, N, ld = packed.shape
    B = BH // heads
    dt = _dtype_code(packed)
    if d_packed is None:
        d_packed = torch.zeros_like(packed)
    vlo, vhi = view_of(do_lo4), view_of(do_hi4)
    nbytes = psa_attn_bwd_ex_workspace_bytes(vlo, vhi, B, heads, N, d, dt, algo)
    ws = (workspace or BwdWorkspace(packed.device)).get(nbytes)
    psa_attn_bwd_ex(packed, ld, o_lo, o_hi, o_lo.shape[-1], lse, vlo, vhi, d_packed, ws, nbytes, B, heads, N, d,
                    scale, dt, algo=algo, stream=stream)
    return d_packed


def merge_bwd(d_merged, heads: int, d: int, stream=None):
    """psa_merge_bwd: d_merged [B, 2*heads*d, H, W] -> (dO_lo, dO_hi) [B*heads, H*W, d]."""
    import torch
    B, c, H, W = d_merged.shape
    d_lo = torch.empty((B * heads, H * W, d), dtype=d_merged.dtype, device=d_merged.device)
    d_hi = torch.empty_like(d_lo)
    psa_merge_bwd(d_merged, d_lo, d_hi, B, heads, H, W, d, _dtype_code(d_merged), stream=stream)
    return d_lo, d_hi


def merge_attn_bwd(packed, o_lo, o_hi, lse, d_merged, heads: int, scale: float, d_packed=None, workspace=None,
                   algo=PSA_ALGO_AUTO, stream=None):
    """psa_merge_attn_bwd: the merge's backward fused into the attention
    backward; d_merged [B, 2*heads*d, H, W].  Returns d_packed."""
    import torch
    BH, _, N, d = packed.shape
    B, c, H, W = d_merged.shape
    dt = _dtype_code(packed)
    if d_packed is None:
        d_packed = torch.empty_like(packed)
    nbytes = psa_merge_attn_bwd_workspace_bytes(B, heads, H, W, d, dt, algo)
    ws = (workspace or BwdWorkspace(packed.device)).get(nbytes)
    psa_merge_attn_bwd(packed, o_lo, o_hi, lse, d_merged, d_packed, ws, nbytes, B, heads, H, W, d, scale, dt,
                       algo=algo, stream=stream)
    return d_packed
