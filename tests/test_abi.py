"""The C ABI library without a GPU: it loads, exports every entry point the
header declares, sizes workspaces, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ncattn.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nc_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    b = __graft_entry__._build_module()
    b.build()
    return ctypes.CDLL(b.LIB)


def test_header_declares_the_three_attention_calls():
    names = _declared()
    for n in ("nc_attn_fwd", "nc_attn_bwd", "nc_attn_decode"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_lists_every_declared_symbol():
    import causal_attention_rope_nc_b300 as nc
    assert sorted(nc.EXPORTED) == _declared()


def test_workspace_sizes(lib):
    f = lib.nc_attn_workspace_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 5
    B, T, H, D = 32, 2048, 10, 128
    tab = T * (D // 2) * 8
    assert f(0, B, T, H, D) == tab
    assert f(1, B, T, H, D) == tab + 2 * B * H * T * 4 + 256
    assert f(2, B, T, H, D) > 0
    assert f(0, B, T, H, 96) == 0  # unsupported head dim


def _fwd(lib):
    f = lib.nc_attn_fwd
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P] * 10 + [ctypes.c_size_t, I, I, I, I, F, F, P]
    f.restype = I
    return f


def test_host_validation_rejects_bad_arguments(lib):
    f = _fwd(lib)
    fake = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
    args = [fake] * 3 + [None] + [fake] * 2 + [fake] * 2 + [None] + [fake]
    ws = 1 << 30
    assert f(*args, ws, 1, 128, 2, 96, 1e-6, 1e4, None) == -1          # D not 64/128
    assert f(*args, ws, 1, 128, 2, 64, -1.0, 1e4, None) == -1          # eps < 0
    assert f(*args, ws, 1, 128, 2, 64, 1e-6, 0.0, None) == -1          # base <= 0
    assert f(*args, ws, -1, 128, 2, 64, 1e-6, 1e4, None) == -1         # negative size
    bad = list(args)
    bad[0] = None
    assert f(*bad, ws, 1, 128, 2, 64, 1e-6, 1e4, None) == -1           # null q
    bad = list(args)
    bad[1] = ctypes.c_void_p(4096 + 2)
    assert f(*bad, ws, 1, 128, 2, 64, 1e-6, 1e4, None) == -1           # misaligned k
    assert f(*args, 16, 1, 128, 2, 64, 1e-6, 1e4, None) == -1          # workspace too small


def test_window_calls_reject_a_negative_window(lib):
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    fake = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
    f = lib.nc_attn_fwd_sw
    f.argtypes = [P] * 10 + [SZ, I, I, I, I, F, F, I, P]
    f.restype = I
    args = [fake] * 3 + [None] + [fake] * 4 + [None] + [fake]
    assert f(*args, 1 << 30, 1, 128, 2, 64, 1e-6, 1e4, -1, None) == -1
    assert f(*([None] * 10), 0, 0, 128, 2, 64, 1e-6, 1e4, 32, None) == 0  # empty problem, any window
    g = lib.nc_attn_bwd_sw
    g.argtypes = [P] * 13 + [SZ, I, I, I, I, F, F, I, P]
    g.restype = I
    assert g(*([fake] * 3 + [None] + [fake] * 9), 1 << 30, 1, 128, 2, 64, 1e-6, 1e4, -5, None) == -1
    d = lib.nc_attn_decode_sw
    d.argtypes = [P] * 8 + [SZ, I, I, I, I, F, F, I, P]
    d.restype = I
    assert d(fake, None, None, fake, fake, fake, fake, fake, 1 << 30, 2, 2, 128, 64, 1e-6, 1e4, -1, None) == -1


def test_empty_problem_is_a_no_op(lib):
    f = _fwd(lib)
    assert f(*([None] * 10), 0, 0, 128, 2, 64, 1e-6, 1e4, None) == 0
    assert f(*([None] * 10), 0, 4, 0, 2, 128, 1e-6, 1e4, None) == 0


def test_decode_rejects_half_given_new_token(lib):
    f = lib.nc_attn_decode
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P] * 8 + [ctypes.c_size_t, I, I, I, I, F, F, P]
    f.restype = I
    fake = ctypes.c_void_p(4096)
    # k_new given, v_new missing
    assert f(fake, fake, None, fake, fake, fake, fake, fake, 1 << 30, 2, 2, 128, 64, 1e-6, 1e4, None) == -1
    # too many heads for one CTA per chunk
    assert f(fake, None, None, fake, fake, fake, fake, fake, 1 << 40, 2, 4096, 128, 64, 1e-6, 1e4, None) == -1


def test_strerror(lib):
    lib.nc_strerror.restype = ctypes.c_char_p
    assert lib.nc_strerror(0) == b"ok"
    assert b"invalid" in lib.nc_strerror(-1)
