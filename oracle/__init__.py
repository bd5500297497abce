"""fp64 CPU oracle for causal attention with QK RMSNorm and RoPE.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path never
imports this package.  The arithmetic lives in ``ncattn_oracle.c`` (plain
loops in double precision); this module only marshals numpy arrays to it.

Every function takes and returns float64 numpy arrays, [B, T, H, D] layout
for token tensors (k, v and their gradients with Hkv <= H heads: grouped-query
attention, query head h using key/value head h // (H // Hkv)), [B, H, T] for
the log-sum-exp.  ``window`` W > 0 restricts
the causal mask to the last W keys (query i sees key j when 0 <= i - j < W);
0 means the plain causal mask.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ncattn_oracle.c")
_LIB = os.path.join(_HERE, "libncattn_oracle.so")

NORM = 1
ROPE = 2
METHOD = NORM | ROPE  # the method: QK RMSNorm and RoPE both applied


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math) in place."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-o", _LIB, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        i, d = ctypes.c_int, ctypes.c_double
        lib.orc_norm_rope.argtypes = [dp, ip, i, i, i, i, d, d, i, dp, dp]
        lib.orc_norm_rope.restype = None
        lib.orc_attn_fwd.argtypes = [dp, dp, dp, ip, i, i, i, i, i, d, d, i, i, dp, dp]
        lib.orc_attn_fwd.restype = ctypes.c_int
        lib.orc_attn_bwd.argtypes = [dp, dp, dp, dp, ip, i, i, i, i, i, d, d, i, i, dp, dp, dp]
        lib.orc_attn_bwd.restype = ctypes.c_int
        lib.orc_attn_decode.argtypes = [dp, dp, dp, ip, i, i, i, i, i, d, d, i, i, dp]
        lib.orc_attn_decode.restype = ctypes.c_int
        lib.orc_attn_prefill.argtypes = [dp, dp, dp, ip, i, i, i, i, i, i, d, d, i, i, dp, dp]
        lib.orc_attn_prefill.restype = ctypes.c_int
        lib.orc_attn_fwd_fp8.argtypes = [dp, dp, dp, ip, i, i, i, i, i, d, d, i, i, dp, dp]
        lib.orc_attn_fwd_fp8.restype = ctypes.c_int
        lib.orc_e4m3.argtypes = [d]
        lib.orc_e4m3.restype = d
        _lib = lib
    return _lib


def _check_groups(H, Hkv, Hv):
    if Hkv != Hv or Hkv < 1 or H % Hkv:
        raise ValueError("key and value heads must match and divide the query heads")


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor (bf16 converts to fp64 exactly)
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _pos(pos, T):
    if pos is None:
        return None, None
    p = np.ascontiguousarray(np.asarray(pos, dtype=np.int32).reshape(T))
    return p, p.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def norm_rope(x, pos=None, eps=1e-6, base=10000.0, flags=METHOD):
    """Normalised and rotated vectors xhat [B,T,H,D] and RMS factors r [B,T,H]."""
    x = _f64(x)
    B, T, H, D = x.shape
    xhat = np.empty_like(x)
    r = np.empty((B, T, H), dtype=np.float64)
    p, pp = _pos(pos, T)
    _load().orc_norm_rope(_dp(x), pp, B, T, H, D, eps, base, flags, _dp(xhat), _dp(r))
    return xhat, r


def attn_fwd(q, k, v, pos=None, eps=1e-6, base=10000.0, flags=METHOD, window=0):
    """Causal attention forward: (o [B,T,H,D], lse [B,H,T])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, T, H, D = q.shape
    o = np.empty_like(q)
    lse = np.empty((B, H, T), dtype=np.float64)
    p, pp = _pos(pos, T)
    Hkv = k.shape[2]
    _check_groups(H, Hkv, v.shape[2])
    rc = _load().orc_attn_fwd(_dp(q), _dp(k), _dp(v), pp, B, T, H, Hkv, D, eps, base, flags, int(window),
                              _dp(o), _dp(lse))
    if rc != 0:
        raise MemoryError("oracle forward failed")
    return o, lse


def attn_bwd(q, k, v, dout, pos=None, eps=1e-6, base=10000.0, flags=METHOD, window=0):
    """Causal attention backward: (dq, dk, dv), each [B,T,H,D]."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, T, H, D = q.shape
    Hkv = k.shape[2]
    _check_groups(H, Hkv, v.shape[2])
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    p, pp = _pos(pos, T)
    rc = _load().orc_attn_bwd(_dp(q), _dp(k), _dp(v), _dp(dout), pp, B, T, H, Hkv, D, eps, base,
                              flags, int(window), _dp(dq), _dp(dk), _dp(dv))
    if rc != 0:
        raise MemoryError("oracle backward failed")
    return dq, dk, dv


def attn_decode(q, k_raw, v, lens, eps=1e-6, base=10000.0, flags=METHOD, window=0):
    """Single-token decode: out [B,H,D] for new queries q [B,H,D] at position
    lens-1 over raw keys k_raw and values v [B,Tcap,H,D]."""
    q, k_raw, v = _f64(q), _f64(k_raw), _f64(v)
    B, Tcap, Hkv, D = k_raw.shape
    H = q.shape[1]
    _check_groups(H, Hkv, v.shape[2])
    lens = np.ascontiguousarray(np.asarray(lens, dtype=np.int32).reshape(B))
    out = np.empty((B, H, D), dtype=np.float64)
    rc = _load().orc_attn_decode(_dp(q), _dp(k_raw), _dp(v),
                                 lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                 B, H, Hkv, D, Tcap, eps, base, flags, int(window), _dp(out))
    if rc != 0:
        raise ValueError("oracle decode: lens out of [1, Tcap]")
    return out


def attn_prefill(q, k_raw, v, start, eps=1e-6, base=10000.0, flags=METHOD, window=0):
    """Prefill of a chunk: (out [B,C,H,D], lse [B,H,C]) for the C new queries
    q [B,C,H,D] of stream b at positions start[b] .. start[b]+C-1, over raw
    keys k_raw and values v [B,Tcap,Hkv,D] (the chunk's own keys and values in
    their slots; Hkv < H: grouped-query attention)."""
    q, k_raw, v = _f64(q), _f64(k_raw), _f64(v)
    B, C, H, D = q.shape
    Tcap, Hkv = k_raw.shape[1], k_raw.shape[2]
    _check_groups(H, Hkv, v.shape[2])
    start = np.ascontiguousarray(np.asarray(start, dtype=np.int32).reshape(B))
    out = np.empty((B, C, H, D), dtype=np.float64)
    lse = np.empty((B, H, C), dtype=np.float64)
    rc = _load().orc_attn_prefill(_dp(q), _dp(k_raw), _dp(v), start.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                  B, C, H, Hkv, D, Tcap, eps, base, flags, int(window), _dp(out), _dp(lse))
    if rc != 0:
        raise ValueError("oracle prefill: start + C outside [0, Tcap]")
    return out, lse



def e4m3(x) -> np.ndarray:
    """The oracle's E4M3 rounding (ties to even, saturating at +-448),
    elementwise."""
    a = _f64(x)
    f = _load().orc_e4m3
    return np.vectorize(f, otypes=[np.float64])(a) if a.size else a.copy()


def attn_fwd_fp8(q, k, v, pos=None, eps=1e-6, base=10000.0, window=0, quant=True):
    """FP8 forward under this library's quantisation reading (see
    orc_attn_fwd_fp8): (o [B,T,H,D], lse [B,H,T]).  quant=False is the plain
    forward."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, T, H, D = q.shape
    o = np.empty_like(q)
    lse = np.empty((B, H, T), dtype=np.float64)
    p, pp = _pos(pos, T)
    Hkv = k.shape[2]
    _check_groups(H, Hkv, v.shape[2])
    rc = _load().orc_attn_fwd_fp8(_dp(q), _dp(k), _dp(v), pp, B, T, H, Hkv, D, eps, base, int(window),
                                  1 if quant else 0, _dp(o), _dp(lse))
    if rc != 0:
        raise MemoryError("oracle fp8 forward failed")
    return o, lse
