"""Pins for the oracle's sliding-window mask (query i sees key j exactly when
0 <= i - j < W): facts fixed by that definition, not by the oracle itself.
The window of the short-window layers is a quarter of the context
(ai.flicky.cc, "nanochat: свой ChatGPT от токенизатора до чата", section
"Модель: что изменилось со времён GPT-2", window-pattern bullet); the
boundary convention (W keys, the query's own included) is this build's
reading of it.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import decode_inputs


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _band(T, W):
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    return (j <= i) & (i - j < W)


@pytest.mark.parametrize("W", [37, 38, 1000])
def test_window_at_least_T_is_plain_causal(W):
    """A window that covers every earlier position changes nothing."""
    B, T, H, D = 2, 37, 2, 16
    q, k, v = (_rand((B, T, H, D), s) for s in (1, 2, 3))
    o0, l0 = oracle.attn_fwd(q, k, v)
    o1, l1 = oracle.attn_fwd(q, k, v, window=W)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_window_one_returns_v():
    """W = 1: every query sees only its own key, so out = v exactly and the
    lse is that single scaled score."""
    B, T, H, D = 2, 23, 3, 8
    q, k, v = (_rand((B, T, H, D), s) for s in (4, 5, 6))
    o, lse = oracle.attn_fwd(q, k, v, window=1, flags=0)
    assert np.array_equal(o, v)
    s = np.einsum("bthd,bthd->bht", q, k) / np.sqrt(D)
    assert np.allclose(lse, s, atol=1e-13)


@pytest.mark.parametrize("W", [1, 5, 16])
def test_plain_windowed_attention_matches_torch_sdpa_band_mask(W):
    """Norm and RoPE off: the forward is SDPA with the band as an explicit
    boolean mask (torch, float64, CPU), and the backward is its autograd."""
    B, T, H, D = 2, 41, 2, 8
    q, k, v, do = (_rand((B, T, H, D), s) for s in (7, 8, 9, 10))
    o, _ = oracle.attn_fwd(q, k, v, flags=0, window=W)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, flags=0, window=W)
    mask = torch.from_numpy(_band(T, W))
    tq, tk, tv = (torch.from_numpy(a).permute(0, 2, 1, 3).clone().requires_grad_() for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)
    assert np.allclose(o, ref.detach().permute(0, 2, 1, 3).numpy(), atol=1e-12)
    ref.backward(torch.from_numpy(do).permute(0, 2, 1, 3))
    for mine, t in ((dq, tq), (dk, tk), (dv, tv)):
        assert np.allclose(mine, t.grad.permute(0, 2, 1, 3).numpy(), atol=1e-12)


def test_keys_outside_the_window_do_not_matter():
    """Changing keys and values at j <= i - W leaves row i unchanged
    (bit-exact), while changing the oldest key inside the window does not."""
    B, T, H, D, W = 1, 30, 2, 8, 6
    q, k, v = (_rand((B, T, H, D), s) for s in (11, 12, 13))
    i = 20
    o1, _ = oracle.attn_fwd(q, k, v, window=W)
    k2, v2 = k.copy(), v.copy()
    k2[:, : i - W + 1] += 3.0
    v2[:, : i - W + 1] -= 2.0
    o2, _ = oracle.attn_fwd(q, k2, v2, window=W)
    assert np.array_equal(o1[:, i], o2[:, i])
    v3 = v.copy()
    v3[:, i - W + 1] += 1.0
    o3, _ = oracle.attn_fwd(q, k, v3, window=W)
    assert not np.array_equal(o1[:, i], o3[:, i])


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


@pytest.mark.parametrize("T,D,W", [(7, 4, 3), (9, 6, 2)])
def test_windowed_backward_matches_finite_differences(T, D, W):
    B, H = 1, 1
    q, k, v, do = (_rand((B, T, H, D), 20 + s) for s in range(4))

    def loss(qq, kk, vv):
        o, _ = oracle.attn_fwd(qq, kk, vv, window=W)
        return float(np.sum(o * do))

    dq, dk, dv = oracle.attn_bwd(q, k, v, do, window=W)
    for mine, fd in ((dq, _fd_grad(lambda x: loss(x, k, v), q)),
                     (dk, _fd_grad(lambda x: loss(q, x, v), k)),
                     (dv, _fd_grad(lambda x: loss(q, k, x), v))):
        rel = np.linalg.norm(mine - fd) / np.linalg.norm(fd)
        assert rel < 1e-6, rel


def test_windowed_gradient_invariant():
    """Rows of P still sum to one: sum_j dv_j = sum_i do_i."""
    B, T, H, D = 2, 33, 2, 16
    q, k, v, do = (_rand((B, T, H, D), 30 + s) for s in range(4))
    _, _, dv = oracle.attn_bwd(q, k, v, do, window=7)
    assert np.allclose(dv.sum(axis=1), do.sum(axis=1), atol=1e-11)


def test_windowed_decode_equals_last_row_of_windowed_forward():
    lens, q, k_raw, v = decode_inputs(B=4, H=3, D=32, Tcap=40, seed=62, lens=[1, 17, 40, 25])
    W = 9
    out = oracle.attn_decode(q, k_raw, v, lens, window=W)
    for b, L in enumerate(lens.tolist()):
        qf = k_raw[b:b + 1, :L].clone()
        qf[0, L - 1] = q[b]
        o, _ = oracle.attn_fwd(qf, k_raw[b:b + 1, :L], v[b:b + 1, :L], window=W)
        assert np.allclose(out[b], o[0, L - 1], atol=1e-13)
