"""Pins for the oracle's grouped-query attention (Hkv key/value heads shared by
groups of H / Hkv consecutive query heads; ai.flicky.cc, "nanochat: свой
ChatGPT от токенизатора до чата", section "Модель: что изменилось со времён
GPT-2", GQA bullet): it must equal multi-head attention on key/value heads
repeated over each group, with the key/value gradients summed over the group.
"""
import numpy as np
import pytest

import oracle
from workloads import decode_inputs


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _rep(x, G):
    return np.repeat(x, G, axis=2)  # head hk -> heads hk*G .. hk*G+G-1


@pytest.mark.parametrize("H,Hkv,W", [(4, 2, 0), (6, 1, 0), (4, 4, 0), (6, 3, 5)])
def test_gqa_equals_mha_with_repeated_heads(H, Hkv, W):
    B, T, D = 2, 19, 16
    G = H // Hkv
    q = _rand((B, T, H, D), 1)
    k, v = _rand((B, T, Hkv, D), 2), _rand((B, T, Hkv, D), 3)
    do = _rand((B, T, H, D), 4)
    o, lse = oracle.attn_fwd(q, k, v, window=W)
    o_r, lse_r = oracle.attn_fwd(q, _rep(k, G), _rep(v, G), window=W)
    assert np.allclose(o, o_r, atol=1e-13) and np.allclose(lse, lse_r, atol=1e-13)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, window=W)
    dq_r, dk_r, dv_r = oracle.attn_bwd(q, _rep(k, G), _rep(v, G), do, window=W)
    assert np.allclose(dq, dq_r, atol=1e-12)
    assert np.allclose(dk, dk_r.reshape(B, T, Hkv, G, D).sum(axis=3), atol=1e-12)
    assert np.allclose(dv, dv_r.reshape(B, T, Hkv, G, D).sum(axis=3), atol=1e-12)


def _fd_grad(f, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        g[idx] = (f(xp) - f(xm)) / (2 * h)
    return g


def test_gqa_backward_matches_finite_differences():
    B, T, H, Hkv, D = 1, 6, 4, 2, 4
    q, do = _rand((B, T, H, D), 10), _rand((B, T, H, D), 11)
    k, v = _rand((B, T, Hkv, D), 12), _rand((B, T, Hkv, D), 13)

    def loss(qq, kk, vv):
        o, _ = oracle.attn_fwd(qq, kk, vv)
        return float(np.sum(o * do))

    dq, dk, dv = oracle.attn_bwd(q, k, v, do)
    for mine, fd in ((dq, _fd_grad(lambda x: loss(x, k, v), q)),
                     (dk, _fd_grad(lambda x: loss(q, x, v), k)),
                     (dv, _fd_grad(lambda x: loss(q, k, x), v))):
        assert np.linalg.norm(mine - fd) / np.linalg.norm(fd) < 1e-6


def test_gqa_decode_equals_repeated_cache():
    lens, _, k_raw, v = decode_inputs(B=3, H=2, D=32, Tcap=30, seed=14, lens=[1, 17, 30])
    q = np.random.default_rng(15).standard_normal((3, 6, 32))
    out = oracle.attn_decode(q, k_raw, v, lens)
    kr = np.repeat(k_raw.double().numpy(), 3, axis=2)
    vr = np.repeat(v.double().numpy(), 3, axis=2)
    assert np.allclose(out, oracle.attn_decode(q, kr, vr, lens), atol=1e-13)


def test_gqa_rejects_heads_that_do_not_divide():
    with pytest.raises(ValueError):
        oracle.attn_fwd(_rand((1, 4, 5, 8), 1), _rand((1, 4, 2, 8), 2), _rand((1, 4, 2, 8), 3))


@pytest.mark.parametrize("W", [0, 7])
def test_gqa_prefill_equals_repeated_cache_and_forward_rows(W):
    """A chunk with Hkv < H key/value heads: the MHA prefill over the heads
    repeated per group, and rows start .. start+C-1 of the GQA forward over
    the whole sequence."""
    B, C, H, Hkv, D, Tcap = 2, 5, 6, 2, 16, 24
    start = [0, 11]
    q = _rand((B, C, H, D), 20)
    k, v = _rand((B, Tcap, Hkv, D), 21), _rand((B, Tcap, Hkv, D), 22)
    out, lse = oracle.attn_prefill(q, k, v, start, window=W)
    out_r, lse_r = oracle.attn_prefill(q, _rep(k, H // Hkv), _rep(v, H // Hkv), start, window=W)
    assert np.allclose(out, out_r, atol=1e-13) and np.allclose(lse, lse_r, atol=1e-13)
    for b, s in enumerate(start):
        T = s + C
        qf = _rand((1, T, H, D), 23)
        qf[0, s:] = q[b]
        o_f, lse_f = oracle.attn_fwd(qf, k[b:b + 1, :T], v[b:b + 1, :T], window=W)
        assert np.allclose(out[b], o_f[0, s:], atol=1e-12)
        assert np.allclose(lse[b], lse_f[0, :, s:], atol=1e-12)


@pytest.mark.parametrize("W", [1, 6, 40])
def test_gqa_windowed_decode_is_the_last_row_of_the_windowed_forward(W):
    """Decode at position L-1 with a window and grouped heads equals row L-1
    of the forward over the prefix with the same window and heads (W = 40
    covers the whole prefix: the plain causal row)."""
    B, H, Hkv, D, L = 1, 6, 2, 16, 23
    q = _rand((B, L, H, D), 30)
    k, v = _rand((B, L, Hkv, D), 31), _rand((B, L, Hkv, D), 32)
    o_f, _ = oracle.attn_fwd(q, k, v, window=W)
    o_d = oracle.attn_decode(q[:, L - 1], k, v, np.array([L], dtype=np.int32), window=W)
    assert np.allclose(o_d, o_f[:, L - 1], atol=1e-12)
