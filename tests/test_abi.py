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


def test_checked_build_exports_every_declared_symbol():
    """The bounds-checked debug build (-DNC_CHECK) has the same ABI."""
    import __graft_entry__
    b = __graft_entry__._build_module()
    chk = ctypes.CDLL(b.build(checked=True))
    for name in _declared():
        assert hasattr(chk, name), name


def test_binding_lists_every_declared_symbol():
    import causal_attention_rope_nc_b300 as nc
    assert sorted(nc.EXPORTED) == _declared()


def test_workspace_sizes(lib):
    f = lib.nc_attn_workspace_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 5
    B, T, H, D = 32, 2048, 10, 128
    tab = T * (D // 2) * 8
    assert f(0, B, T, H, D) == tab + 256  # RoPE table, the forward's pair counter
    n_t = T // 128
    assert f(1, B, T, H, D) == tab + 2 * B * H * T * 4 + 256 + B * H * (n_t * (n_t + 1) // 2) * 128 * 128 * 2
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


def _ex_calls(lib):
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    f = lib.nc_attn_fwd_ex
    f.argtypes = [P] * 10 + [SZ, I, I, I, I, F, F, I, I, P]
    f.restype = I
    g = lib.nc_attn_bwd_ex
    g.argtypes = [P] * 13 + [SZ, I, I, I, I, F, F, I, I, P]
    g.restype = I
    d = lib.nc_attn_decode_ex
    d.argtypes = [P] * 8 + [SZ, I, I, I, I, F, F, I, I, P]
    d.restype = I
    pf = lib.nc_attn_prefill
    pf.argtypes = [P] * 9 + [SZ, I, I, I, I, I, F, F, I, I, P]
    pf.restype = I
    return f, g, d, pf


def test_ex_calls_reject_a_negative_window(lib):
    f, g, d, _ = _ex_calls(lib)
    fake = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
    args = [fake] * 3 + [None] + [fake] * 4 + [None] + [fake]
    assert f(*args, 1 << 30, 1, 128, 2, 64, 1e-6, 1e4, -1, 0, None) == -1
    assert f(*([None] * 10), 0, 0, 128, 2, 64, 1e-6, 1e4, 32, 0, None) == 0  # empty problem, any window
    assert g(*([fake] * 3 + [None] + [fake] * 9), 1 << 30, 1, 128, 2, 64, 1e-6, 1e4, -5, 0, None) == -1
    assert d(fake, None, None, fake, fake, fake, fake, fake, 1 << 30, 2, 2, 128, 64, 1e-6, 1e4, -1, 0, None) == -1


def test_ex_calls_reject_kv_heads_that_do_not_divide_h(lib):
    """Grouped-query attention: kv_heads must divide H (0 means H)."""
    f, g, d, pf = _ex_calls(lib)
    fake = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
    args = [fake] * 3 + [None] + [fake] * 4 + [None] + [fake]
    for bad in (-1, 3, 8, 5):  # H = 4
        assert f(*args, 1 << 30, 1, 128, 4, 64, 1e-6, 1e4, 0, bad, None) == -1, bad
        assert g(*([fake] * 3 + [None] + [fake] * 9), 1 << 30, 1, 128, 4, 64, 1e-6, 1e4, 0, bad, None) == -1
        assert d(fake, None, None, fake, fake, fake, fake, fake, 1 << 30, 2, 4, 64, 128, 1e-6, 1e4, 0, bad,
                 None) == -1
        assert pf(*([fake] * 9), 1 << 30, 1, 128, 4, 64, 256, 1e-6, 1e4, 0, bad, None) == -1
        # the head check comes before the empty-problem shortcut
        assert f(*([None] * 10), 0, 0, 128, 4, 64, 1e-6, 1e4, 0, bad, None) == -1
    for ok in (0, 1, 2, 4):  # divisors of H = 4 (0 meaning H): an empty problem is a no-op
        assert f(*([None] * 10), 0, 0, 128, 4, 64, 1e-6, 1e4, 0, ok, None) == 0
        assert g(*([None] * 13), 0, 0, 128, 4, 64, 1e-6, 1e4, 0, ok, None) == 0


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


def test_binding_checks_grouped_heads_on_the_host():
    """The binding derives kv_heads from k's shape and refuses a head count
    that does not divide H before any call reaches the library."""
    import torch
    import causal_attention_rope_nc_b300 as nc
    q = torch.empty((1, 4, 6, 64), dtype=torch.bfloat16)
    assert nc._kv_heads(q, torch.empty((1, 4, 3, 64))) == 3
    assert nc._kv_heads(q, torch.empty((1, 4, 6, 64))) == 6
    with pytest.raises(ValueError):
        nc._kv_heads(q, torch.empty((1, 4, 4, 64)))
    with pytest.raises(ValueError):
        nc._shape(torch.empty((1, 4, 2, 64)), "k", (1, 4, 3, 64))
    nc._shape(None, "k_new", (1, 3, 64))  # an absent optional tensor passes


def test_version_names_the_bf16_key_cache(lib):
    """0.3: the key cache is bf16 and the backward keeps a dS scratch (0.2
    added kv_heads)."""
    lib.nc_version.restype = ctypes.c_int
    assert lib.nc_version() == (0 << 16) | 3


def test_binding_rejects_wrong_16bit_types():
    """The binding refuses a key cache that is not bf16, and qhat or khat
    that are not fp16, before the C call."""
    import torch
    import causal_attention_rope_nc_b300 as nc
    with pytest.raises(ValueError, match="bfloat16"):
        nc._bf16(torch.empty((1, 4, 2, 64), dtype=torch.float16), "kcache")
    with pytest.raises(ValueError, match="float16"):
        nc._f16(torch.empty((1, 4, 2, 64), dtype=torch.bfloat16), "qhat")

