"""B300 (sm_103a) causal attention with QK RMSNorm and RoPE -- Python binding.

This module only marshals torch tensors to the C ABI of ``libncattn.so``
(declared in ``include/ncattn.h``); every step of the computation runs in the
library's CUDA kernels.  There is no CPU fallback: if the library is missing
the import fails, and every call checks the status the library returns.

The functions named ``nc_*`` mirror the C entry points one to one (torch
tensors in place of pointers, the current CUDA stream by default).  The
``attn_*`` helpers allocate outputs and workspaces with torch and call them:

    out, lse, qhat, khat = attn_fwd(q, k, v)            # q, k, v [B, T, H, D] bf16, CUDA (qhat, khat fp16)
    dq, dk, dv = attn_bwd(q, k, v, out, lse, qhat, khat, dout)
    out, lse, qhat, khat = attn_fwd(q, k, v, window=512)  # sliding window
    out, lse, qhat, khat = attn_fwd(q, k2, v2)           # k2, v2 [B, T, 2, D]: 2 key/value heads
    kcache = qk_norm_rope(k_prompt)                      # prefill a key cache [B, Tcap, Hkv, D] (bf16)
    o = attn_decode(q1, kcache, vcache, lens, k_new=k1, v_new=v1)   # one new token per stream
    out, lse = attn_prefill(qc, kc, vc, start, kcache, vcache)      # a chunk at offsets start[b]
    out, lse = attn_fwd_fp8(q, k, v)                     # E4M3 products (head dim 128)

Grouped-query attention needs no flag: the key/value heads are read from k's
(or the cache's) shape and must divide H.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libncattn.so")

NC_OK, NC_EINVAL, NC_EUNSUPPORTED, NC_ELAUNCH, NC_EDEVICE = 0, -1, -2, -3, -4
NC_OP_FWD, NC_OP_BWD, NC_OP_DECODE, NC_OP_NORM_ROPE, NC_OP_PREFILL, NC_OP_FWD_FP8 = 0, 1, 2, 3, 4, 5

EXPORTED = ("nc_version", "nc_strerror", "nc_last_cuda_error", "nc_device_status",
            "nc_attn_workspace_size", "nc_qk_norm_rope", "nc_attn_fwd", "nc_attn_bwd",
            "nc_attn_decode", "nc_profile_enable", "nc_profile_read", "nc_attn_decode_noalloc",
            "nc_attn_fwd_ex", "nc_attn_bwd_ex", "nc_attn_decode_ex", "nc_attn_prefill", "nc_attn_fwd_fp8")
NC_ETOOLARGE = -5


class NcError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        extra = ""
        if code == NC_ELAUNCH:
            extra = f" (cudaError {lib.nc_last_cuda_error()})"
        super().__init__(f"{what}: {lib.nc_strerror(code).decode()} [{code}]{extra}")


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int), ("kernels", ctypes.c_int),
                ("total_ms", ctypes.c_double)]


LIB_CHECK_PATH = os.path.join(_HERE, "libncattn_check.so")


def _load(path=None):
    """The library's ctypes handle with every entry point typed.  path:
    LIB_PATH by default; LIB_CHECK_PATH gives the bounds-checked debug build
    (same entry points), which the bounds tests load beside the normal one."""
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(path)
    P, I, F, S, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
    L.nc_version.restype = I
    L.nc_strerror.argtypes = [I]
    L.nc_strerror.restype = ctypes.c_char_p
    L.nc_last_cuda_error.restype = I
    L.nc_device_status.argtypes = [S, ctypes.POINTER(ctypes.c_uint)]
    L.nc_device_status.restype = I
    L.nc_attn_workspace_size.argtypes = [I, I, I, I, I]
    L.nc_attn_workspace_size.restype = SZ
    L.nc_qk_norm_rope.argtypes = [P, P, P, P, P, SZ, I, I, I, I, F, F, S]
    L.nc_qk_norm_rope.restype = I
    L.nc_attn_fwd.argtypes = [P, P, P, P, P, P, P, P, P, P, SZ, I, I, I, I, F, F, S]
    L.nc_attn_fwd.restype = I
    L.nc_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, I, I, I, I, F, F, S]
    L.nc_attn_bwd.restype = I
    L.nc_attn_decode.argtypes = [P, P, P, P, P, P, P, P, SZ, I, I, I, I, F, F, S]
    L.nc_attn_decode.restype = I
    L.nc_profile_enable.argtypes = [I]
    L.nc_profile_enable.restype = I
    L.nc_profile_read.argtypes = [ctypes.POINTER(KernelTime), I, ctypes.POINTER(I)]
    L.nc_profile_read.restype = I
    L.nc_attn_decode_noalloc.argtypes = [P, P, P, P, P, P, P, I, I, I, I, F, F, S]
    L.nc_attn_decode_noalloc.restype = I
    L.nc_attn_fwd_ex.argtypes = [P, P, P, P, P, P, P, P, P, P, SZ, I, I, I, I, F, F, I, I, S]
    L.nc_attn_fwd_ex.restype = I
    L.nc_attn_bwd_ex.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, I, I, I, I, F, F, I, I, S]
    L.nc_attn_bwd_ex.restype = I
    L.nc_attn_decode_ex.argtypes = [P, P, P, P, P, P, P, P, SZ, I, I, I, I, F, F, I, I, S]
    L.nc_attn_decode_ex.restype = I
    L.nc_attn_prefill.argtypes = [P, P, P, P, P, P, P, P, P, SZ, I, I, I, I, I, F, F, I, I, S]
    L.nc_attn_prefill.restype = I
    L.nc_attn_fwd_fp8.argtypes = [P, P, P, P, P, P, P, SZ, I, I, I, I, F, F, I, I, S]
    L.nc_attn_fwd_fp8.restype = I
    return L


lib = _load()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(rc: int, what: str):
    if rc != NC_OK:
        raise NcError(rc, what)


def _bf16(t, name, dtype=torch.bfloat16):
    if t is None:
        return
    if t.dtype != dtype or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def _f16(t, name):
    _bf16(t, name, torch.float16)


def workspace_size(op: int, B: int, T: int, H: int, D: int) -> int:
    return int(lib.nc_attn_workspace_size(op, B, T, H, D))


def new_workspace(op: int, B: int, T: int, H: int, D: int, device=None) -> torch.Tensor:
    """Zero-filled workspace (torch allocations are 256-byte aligned)."""
    n = max(workspace_size(op, B, T, H, D), 1)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def device_status(stream=None) -> int:
    st = ctypes.c_uint(0)
    _check(lib.nc_device_status(_stream(stream), ctypes.byref(st)), "nc_device_status")
    return st.value


def nc_profile_enable(on: bool):
    _check(lib.nc_profile_enable(1 if on else 0), "nc_profile_enable")


last_profile_kernels: dict = {}


def nc_profile_read() -> dict:
    """{step name: (timed steps, total ms)} since the last read; the kernel
    launches inside each name's steps go to ``last_profile_kernels``."""
    global last_profile_kernels
    buf = (KernelTime * 64)()
    n = ctypes.c_int(0)
    _check(lib.nc_profile_read(buf, 64, ctypes.byref(n)), "nc_profile_read")
    m = min(n.value, 64)
    last_profile_kernels = {buf[i].name.decode(): buf[i].kernels for i in range(m)}
    return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(m)}


# ------------------------------------------------------ C entry points 1:1 --

def nc_qk_norm_rope(x, pos, xhat, rstd, workspace, eps, rope_base, stream=None):
    _bf16(x, "x"), _bf16(xhat, "xhat")
    B, T, H, D = x.shape
    _check(lib.nc_qk_norm_rope(_ptr(x), _ptr(pos), _ptr(xhat), _ptr(rstd), _ptr(workspace),
                               workspace.numel(), B, T, H, D, eps, rope_base, _stream(stream)),
           "nc_qk_norm_rope")


def _shape(t, name, shape):
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _kv_heads(q, k):
    """Key/value heads of a (q, k) pair: k.shape[2], which must divide H."""
    H, Hkv = q.shape[2], k.shape[2]
    if Hkv < 1 or H % Hkv:
        raise ValueError(f"{Hkv} key/value heads do not divide {H} query heads")
    return Hkv


def _fwd_args(q, k, v, pos, out, lse, qhat, khat, rstd, workspace):
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _bf16(t, n)
    _f16(qhat, "qhat"), _f16(khat, "khat")
    B, T, H, D = q.shape
    Hkv = _kv_heads(q, k)
    for n, t in (("k", k), ("v", v), ("khat", khat)):
        _shape(t, n, (B, T, Hkv, D))
    _shape(out, "out", q.shape), _shape(qhat, "qhat", q.shape)
    return (_ptr(q), _ptr(k), _ptr(v), _ptr(pos), _ptr(out), _ptr(lse), _ptr(qhat), _ptr(khat), _ptr(rstd),
            _ptr(workspace), workspace.numel(), B, T, H, D)


def nc_attn_fwd(q, k, v, pos, out, lse, qhat, khat, rstd, workspace, eps, rope_base, stream=None):
    args = _fwd_args(q, k, v, pos, out, lse, qhat, khat, rstd, workspace)
    if k.shape[2] != q.shape[2]:
        raise ValueError("nc_attn_fwd takes H key/value heads; use nc_attn_fwd_ex for fewer")
    _check(lib.nc_attn_fwd(*args, eps, rope_base, _stream(stream)), "nc_attn_fwd")


def nc_attn_fwd_ex(q, k, v, pos, out, lse, qhat, khat, rstd, workspace, eps, rope_base, window=0, stream=None):
    """kv_heads is k.shape[2] (grouped-query attention when it is below H)."""
    args = _fwd_args(q, k, v, pos, out, lse, qhat, khat, rstd, workspace)
    _check(lib.nc_attn_fwd_ex(*args, eps, rope_base, int(window), k.shape[2], _stream(stream)), "nc_attn_fwd_ex")


def _bwd_args(q, k, v, pos, out, lse, qhat, khat, dout, dq, dk, dv, workspace):
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout), ("dq", dq), ("dk", dk),
                 ("dv", dv)):
        _bf16(t, n)
    _f16(qhat, "qhat"), _f16(khat, "khat")
    B, T, H, D = q.shape
    Hkv = _kv_heads(q, k)
    for n, t in (("k", k), ("v", v), ("khat", khat), ("dk", dk), ("dv", dv)):
        _shape(t, n, (B, T, Hkv, D))
    for n, t in (("out", out), ("qhat", qhat), ("dout", dout), ("dq", dq)):
        _shape(t, n, q.shape)
    return (_ptr(q), _ptr(k), _ptr(v), _ptr(pos), _ptr(out), _ptr(lse), _ptr(qhat), _ptr(khat), _ptr(dout),
            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(), B, T, H, D)


def nc_attn_fwd_fp8(q, k, v, pos, out, lse, workspace, eps, rope_base, window=0, stream=None):
    """FP8 forward (E4M3 products; head dim 128); kv_heads is k.shape[2]."""
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _bf16(t, n)
    B, T, H, D = q.shape
    Hkv = _kv_heads(q, k)
    _shape(k, "k", (B, T, Hkv, D)), _shape(v, "v", (B, T, Hkv, D)), _shape(out, "out", q.shape)
    _shape(lse, "lse", (B, H, T))
    _check(lib.nc_attn_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(pos), _ptr(out), _ptr(lse), _ptr(workspace),
                               workspace.numel(), B, T, H, D, eps, rope_base, int(window), Hkv, _stream(stream)),
           "nc_attn_fwd_fp8")


def nc_attn_bwd(q, k, v, pos, out, lse, qhat, khat, dout, dq, dk, dv, workspace, eps, rope_base,
                stream=None):
    args = _bwd_args(q, k, v, pos, out, lse, qhat, khat, dout, dq, dk, dv, workspace)
    if k.shape[2] != q.shape[2]:
        raise ValueError("nc_attn_bwd takes H key/value heads; use nc_attn_bwd_ex for fewer")
    _check(lib.nc_attn_bwd(*args, eps, rope_base, _stream(stream)), "nc_attn_bwd")


def nc_attn_bwd_ex(q, k, v, pos, out, lse, qhat, khat, dout, dq, dk, dv, workspace, eps, rope_base, window=0,
                   stream=None):
    """kv_heads is k.shape[2] (grouped-query attention when it is below H)."""
    args = _bwd_args(q, k, v, pos, out, lse, qhat, khat, dout, dq, dk, dv, workspace)
    _check(lib.nc_attn_bwd_ex(*args, eps, rope_base, int(window), k.shape[2], _stream(stream)), "nc_attn_bwd_ex")


def _decode_args(q, k_new, v_new, kcache, vcache, lens, out, workspace):
    for n, t in (("q", q), ("k_new", k_new), ("v_new", v_new), ("kcache", kcache), ("vcache", vcache),
                 ("out", out)):
        _bf16(t, n)
    B, Tcap, Hkv, D = kcache.shape
    H = q.shape[1]
    if H % Hkv:
        raise ValueError(f"{Hkv} key/value heads do not divide {H} query heads")
    _shape(q, "q", (B, H, D)), _shape(out, "out", (B, H, D)), _shape(vcache, "vcache", kcache.shape)
    _shape(k_new, "k_new", (B, Hkv, D)), _shape(v_new, "v_new", (B, Hkv, D))
    if lens is None or lens.dtype != torch.int32 or not lens.is_cuda or tuple(lens.shape) != (B,):
        raise ValueError(f"lens must be a CUDA int32 tensor of shape ({B},)")
    return (_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(kcache), _ptr(vcache), _ptr(lens), _ptr(out),
            _ptr(workspace), 0 if workspace is None else workspace.numel(), B, H, D, Tcap)


def nc_attn_decode(q, k_new, v_new, kcache, vcache, lens, out, workspace, eps, rope_base, stream=None):
    args = _decode_args(q, k_new, v_new, kcache, vcache, lens, out, workspace)
    if kcache.shape[2] != q.shape[1]:
        raise ValueError("nc_attn_decode takes H key/value heads; use nc_attn_decode_ex for fewer")
    _check(lib.nc_attn_decode(*args, eps, rope_base, _stream(stream)), "nc_attn_decode")


def nc_attn_decode_ex(q, k_new, v_new, kcache, vcache, lens, out, workspace, eps, rope_base, window=0,
                      stream=None):
    """kv_heads is kcache.shape[2] (grouped-query attention when it is below H)."""
    args = _decode_args(q, k_new, v_new, kcache, vcache, lens, out, workspace)
    _check(lib.nc_attn_decode_ex(*args, eps, rope_base, int(window), kcache.shape[2], _stream(stream)),
           "nc_attn_decode_ex")


def nc_attn_prefill(q, k, v, start, kcache, vcache, out, lse, workspace, eps, rope_base, window=0, stream=None):
    for n, t in (("q", q), ("k", k), ("v", v), ("kcache", kcache), ("vcache", vcache), ("out", out)):
        _bf16(t, n)
    B, C, H, D = q.shape
    Tcap = kcache.shape[1]
    Hkv = _kv_heads(q, k)
    _shape(k, "k", (B, C, Hkv, D)), _shape(v, "v", (B, C, Hkv, D)), _shape(out, "out", q.shape)
    _shape(kcache, "kcache", (B, Tcap, Hkv, D)), _shape(vcache, "vcache", (B, Tcap, Hkv, D))
    _check(lib.nc_attn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(start), _ptr(kcache), _ptr(vcache), _ptr(out),
                               _ptr(lse), _ptr(workspace), workspace.numel(), B, C, H, D, Tcap, eps, rope_base,
                               int(window), Hkv, _stream(stream)), "nc_attn_prefill")


def nc_attn_decode_noalloc(q, k_new, v_new, kcache, vcache, lens, out, eps, rope_base, stream=None):
    """nc_attn_decode for callers that cannot supply a workspace (the library
    keeps the scratch in a fixed 16 MiB device array; see include/ncattn.h).
    Multi-head attention only: the cache has H key/value heads."""
    if kcache.shape[2] != q.shape[1]:
        raise ValueError("nc_attn_decode_noalloc takes H key/value heads (no grouped-query attention)")
    B, H, D, Tcap = _decode_args(q, k_new, v_new, kcache, vcache, lens, out, None)[-4:]
    _check(lib.nc_attn_decode_noalloc(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(kcache), _ptr(vcache),
                                      _ptr(lens), _ptr(out), B, H, D, Tcap, eps, rope_base,
                                      _stream(stream)), "nc_attn_decode_noalloc")


# -------------------------------------------------------- allocating helpers --

def attn_fwd(q, k, v, pos=None, eps=1e-6, rope_base=10000.0, workspace=None, stream=None, window=0):
    """Returns (out, lse, qhat, khat).  window > 0: sliding-window mask; k and
    v with fewer heads than q: grouped-query attention."""
    B, T, H, D = q.shape
    out = torch.empty_like(q)
    qhat = torch.empty_like(q, dtype=torch.float16)
    khat = torch.empty_like(k, dtype=torch.float16)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    ws = workspace if workspace is not None else new_workspace(NC_OP_FWD, B, T, H, D, q.device)
    if window or k.shape[2] != H:
        nc_attn_fwd_ex(q, k, v, pos, out, lse, qhat, khat, None, ws, eps, rope_base, window, stream)
    else:
        nc_attn_fwd(q, k, v, pos, out, lse, qhat, khat, None, ws, eps, rope_base, stream)
    return out, lse, qhat, khat


def attn_fwd_fp8(q, k, v, pos=None, eps=1e-6, rope_base=10000.0, workspace=None, stream=None, window=0):
    """FP8 forward: returns (out, lse); see nc_attn_fwd_fp8 in include/ncattn.h
    for the quantisation."""
    B, T, H, D = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    ws = workspace if workspace is not None else new_workspace(NC_OP_FWD_FP8, B, T, H, D, q.device)
    nc_attn_fwd_fp8(q, k, v, pos, out, lse, ws, eps, rope_base, window, stream)
    return out, lse


def attn_bwd(q, k, v, out, lse, qhat, khat, dout, pos=None, eps=1e-6, rope_base=10000.0,
             workspace=None, stream=None, window=0):
    """Returns (dq, dk, dv) (dk, dv with k's heads).  window: as passed to attn_fwd."""
    B, T, H, D = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = workspace if workspace is not None else new_workspace(NC_OP_BWD, B, T, H, D, q.device)
    if window or k.shape[2] != H:
        nc_attn_bwd_ex(q, k, v, pos, out, lse, qhat, khat, dout, dq, dk, dv, ws, eps, rope_base, window, stream)
    else:
        nc_attn_bwd(q, k, v, pos, out, lse, qhat, khat, dout, dq, dk, dv, ws, eps, rope_base, stream)
    return dq, dk, dv


def qk_norm_rope(x, pos=None, eps=1e-6, rope_base=10000.0, stream=None):
    B, T, H, D = x.shape
    xhat = torch.empty_like(x)
    ws = new_workspace(NC_OP_NORM_ROPE, B, T, H, D, x.device)
    nc_qk_norm_rope(x, pos, xhat, None, ws, eps, rope_base, stream)
    return xhat


def attn_decode(q, kcache, vcache, lens, k_new=None, v_new=None, eps=1e-6, rope_base=10000.0,
                workspace=None, stream=None, window=0):
    B, Tcap, Hkv, D = kcache.shape
    H = q.shape[1]
    out = torch.empty((B, H, D), dtype=torch.bfloat16, device=q.device)
    ws = workspace if workspace is not None else new_workspace(NC_OP_DECODE, B, Tcap, H, D, q.device)
    if window or Hkv != H:
        nc_attn_decode_ex(q, k_new, v_new, kcache, vcache, lens, out, ws, eps, rope_base, window, stream)
    else:
        nc_attn_decode(q, k_new, v_new, kcache, vcache, lens, out, ws, eps, rope_base, stream)
    return out


def attn_prefill(q, k, v, start, kcache, vcache, eps=1e-6, rope_base=10000.0, window=0, workspace=None,
                 stream=None):
    """Chunk prefill: appends the chunk's normalised, rotated keys and its
    values to the caches in place and returns (out [B,C,H,D], lse [B,H,C])."""
    B, C, H, D = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((B, H, C), dtype=torch.float32, device=q.device)
    ws = workspace if workspace is not None else new_workspace(NC_OP_PREFILL, B, C, H, D, q.device)
    nc_attn_prefill(q, k, v, start, kcache, vcache, out, lse, ws, eps, rope_base, window, stream)
    return out, lse

