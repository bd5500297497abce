"""Pins for the fp64 oracle: facts fixed by the definition and the mathematics,
not by the oracle itself.  Each test is chosen so that a plausible slip in the
oracle (a dropped scale, a wrong RoPE sign or pairing, an off-by-one in the
causal mask, a transposed gradient) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from workloads import attn_inputs, decode_inputs


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- softmax ---

def test_softmax_rows_sum_to_one():
    """With every value vector equal to 1, out = sum_j P_ij = 1 for every row."""
    B, T, H, D = 2, 37, 3, 16
    q, k = _rand((B, T, H, D), 1), _rand((B, T, H, D), 2)
    v = np.ones((B, T, H, D))
    o, _ = oracle.attn_fwd(q, k, v)
    assert np.max(np.abs(o - 1.0)) < 1e-12


def test_single_token_returns_v():
    """T = 1: the only key is the query's own, so out = v."""
    q, k, v = _rand((3, 1, 2, 8), 3), _rand((3, 1, 2, 8), 4), _rand((3, 1, 2, 8), 5)
    o, lse = oracle.attn_fwd(q, k, v)
    assert np.array_equal(o, v)


def test_first_row_is_v0():
    """Row 0 attends only to key 0 for any T."""
    B, T, H, D = 2, 19, 2, 8
    q, k, v = _rand((B, T, H, D), 6), _rand((B, T, H, D), 7), _rand((B, T, H, D), 8)
    o, _ = oracle.attn_fwd(q, k, v)
    assert np.array_equal(o[:, 0], v[:, 0])


def test_lse_closed_form_uniform_scores():
    """With q = 0 every score is 0: P is uniform over i+1 keys and
    lse_i = ln(i+1), out_i = mean of v_0..v_i."""
    B, T, H, D = 1, 23, 2, 8
    q = np.zeros((B, T, H, D))
    k, v = _rand((B, T, H, D), 9), _rand((B, T, H, D), 10)
    o, lse = oracle.attn_fwd(q, k, v)
    i = np.arange(T)
    assert np.allclose(lse[0, 0], np.log(i + 1), atol=1e-13)
    ref = np.cumsum(v, axis=1) / (i + 1)[None, :, None, None]
    assert np.allclose(o, ref, atol=1e-13)


# ---------------------------------------------------------------- RMSNorm ---

def test_rmsnorm_closed_form_norm():
    """||x/r||^2 = D * S / (S + D*eps), S = sum x^2; RoPE keeps it."""
    B, T, H, D, eps = 2, 5, 3, 64, 1e-3
    x = _rand((B, T, H, D), 11) * 0.05
    S = np.sum(x * x, axis=-1)
    want = D * S / (S + D * eps)
    for flags in (oracle.NORM, oracle.NORM | oracle.ROPE):
        xh, r = oracle.norm_rope(x, eps=eps, flags=flags)
        assert np.allclose(np.sum(xh * xh, axis=-1), want, rtol=1e-12)
    assert np.allclose(r, np.sqrt(S / D + eps), rtol=1e-14)


def test_rmsnorm_matches_torch_rms_norm():
    """Library special case: parameter-free RMSNorm over the head dim equals
    torch.nn.functional.rms_norm in float64."""
    x = _rand((2, 7, 3, 32), 12)
    xh, _ = oracle.norm_rope(x, eps=1e-6, flags=oracle.NORM)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (32,), eps=1e-6).numpy()
    assert np.allclose(xh, ref, rtol=1e-13, atol=1e-14)


def test_scale_invariance_of_qk_norm():
    """With eps = 0 the method is exactly invariant to positive rescaling of
    q and k per row (the norm removes it)."""
    B, T, H, D = 1, 17, 2, 16
    q, k, v = _rand((B, T, H, D), 13), _rand((B, T, H, D), 14), _rand((B, T, H, D), 15)
    o1, l1 = oracle.attn_fwd(q, k, v, eps=0.0)
    o2, l2 = oracle.attn_fwd(3.7 * q, 0.2 * k, v, eps=0.0)
    assert np.allclose(o1, o2, atol=1e-12) and np.allclose(l1, l2, atol=1e-12)


# ------------------------------------------------------------------- RoPE ---

def test_rope_preserves_norm():
    x = _rand((1, 40, 2, 64), 16)
    xh, _ = oracle.norm_rope(x, flags=oracle.ROPE)
    assert np.allclose(np.linalg.norm(xh, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_two_dims_is_plane_rotation_by_position():
    """D = 2: theta_0 = base^0 = 1, so position p rotates the plane by p rad."""
    x = np.array([0.3, -1.1]).reshape(1, 1, 1, 2)
    for p in (0, 1, 5, 1000):
        xh, _ = oracle.norm_rope(x, pos=[p], flags=oracle.ROPE)
        c, s = math.cos(p), math.sin(p)
        want = [0.3 * c + 1.1 * s, 0.3 * s - 1.1 * c]
        assert np.allclose(xh.reshape(2), want, atol=1e-12)


def test_rope_equals_complex_multiplication():
    """Rotate-half RoPE is the complex product (x_i + i x_{i+D/2}) e^{i p theta_i},
    theta_i = base^(-2i/D): an independent formulation in numpy complex."""
    B, T, H, D, base = 1, 33, 2, 16, 10000.0
    x = _rand((B, T, H, D), 17)
    pos = np.arange(T) * 3 + 5
    xh, _ = oracle.norm_rope(x, pos=pos, base=base, flags=oracle.ROPE)
    z = x[..., : D // 2] + 1j * x[..., D // 2:]
    theta = base ** (-2.0 * np.arange(D // 2) / D)
    zr = z * np.exp(1j * pos[None, :, None, None] * theta)
    assert np.allclose(xh, np.concatenate([zr.real, zr.imag], -1), atol=1e-12)


def test_relative_position_invariance():
    """<R_m q, R_n k> depends on n - m only: shifting every position by a
    constant leaves out and lse unchanged."""
    B, T, H, D = 1, 29, 2, 32
    q, k, v = _rand((B, T, H, D), 18), _rand((B, T, H, D), 19), _rand((B, T, H, D), 20)
    o1, l1 = oracle.attn_fwd(q, k, v)
    o2, l2 = oracle.attn_fwd(q, k, v, pos=np.arange(T) + 777)
    assert np.allclose(o1, o2, atol=1e-11) and np.allclose(l1, l2, atol=1e-11)
    # ...whereas a non-uniform change of positions does change the result
    o3, _ = oracle.attn_fwd(q, k, v, pos=np.arange(T) * 2)
    assert np.max(np.abs(o1 - o3)) > 1e-3


# -------------------------------------------------------------- causality ---

def test_causal_future_does_not_leak():
    B, T, H, D, t0 = 1, 31, 2, 16, 12
    q, k, v = _rand((B, T, H, D), 21), _rand((B, T, H, D), 22), _rand((B, T, H, D), 23)
    o1, l1 = oracle.attn_fwd(q, k, v)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for a, s in ((q2, 24), (k2, 25), (v2, 26)):
        a[:, t0 + 1:] = _rand(a[:, t0 + 1:].shape, s)
    o2, l2 = oracle.attn_fwd(q2, k2, v2)
    assert np.array_equal(o1[:, : t0 + 1], o2[:, : t0 + 1])
    assert np.array_equal(l1[..., : t0 + 1], l2[..., : t0 + 1])
    # the diagonal is included: changing v at t0 changes row t0
    v3 = v.copy()
    v3[:, t0] += 1.0
    o3, _ = oracle.attn_fwd(q, k, v3)
    assert not np.array_equal(o1[:, t0], o3[:, t0])


# --------------------------------------------------- library special case ---

def test_plain_attention_matches_torch_sdpa():
    """With the norm and RoPE switched off the forward is plain causal SDPA
    with scale 1/sqrt(D) (torch, float64, CPU)."""
    B, T, H, D = 2, 45, 3, 16
    q, k, v = _rand((B, T, H, D), 27), _rand((B, T, H, D), 28), _rand((B, T, H, D), 29)
    o, _ = oracle.attn_fwd(q, k, v, flags=0)
    tq, tk, tv = (torch.from_numpy(a).permute(0, 2, 1, 3) for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    assert np.allclose(o, ref.permute(0, 2, 1, 3).numpy(), atol=1e-12)


def test_plain_attention_backward_matches_torch_autograd_sdpa():
    B, T, H, D = 1, 21, 2, 8
    q, k, v, do = (_rand((B, T, H, D), s) for s in (30, 31, 32, 33))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, flags=0)
    tq, tk, tv = (torch.from_numpy(a).permute(0, 2, 1, 3).clone().requires_grad_() for a in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    out.backward(torch.from_numpy(do).permute(0, 2, 1, 3))
    for mine, t in ((dq, tq), (dk, tk), (dv, tv)):
        assert np.allclose(mine, t.grad.permute(0, 2, 1, 3).numpy(), atol=1e-12)


# ---------------------------------------------------------- closed form -----

def test_hand_worked_two_token_example():
    """D = 2, eps = 0, q_t = k_t = (1, 0), positions 0, 1.
    Norm: xhat = (sqrt2, 0).  RoPE (theta_0 = 1): at p = 1 the vector turns by
    1 rad.  Scores of row 1 (scale 1/sqrt2): s10 = 2 cos(1)/sqrt2 = sqrt2 cos 1,
    s11 = 2/sqrt2 = sqrt2.  out_1 = softmax(s10, s11) . (v0, v1)."""
    q = np.array([1.0, 0.0, 1.0, 0.0]).reshape(1, 2, 1, 2)
    k = q.copy()
    v = np.array([2.0, -1.0, 0.5, 4.0]).reshape(1, 2, 1, 2)
    o, lse = oracle.attn_fwd(q, k, v, eps=0.0)
    s10, s11 = math.sqrt(2) * math.cos(1.0), math.sqrt(2)
    p10 = math.exp(s10) / (math.exp(s10) + math.exp(s11))
    want = p10 * v[0, 0, 0] + (1 - p10) * v[0, 1, 0]
    assert np.allclose(o[0, 1, 0], want, atol=1e-14)
    assert math.isclose(lse[0, 0, 1], math.log(math.exp(s10) + math.exp(s11)), abs_tol=1e-14)
    assert math.isclose(lse[0, 0, 0], math.sqrt(2), abs_tol=1e-14)


# -------------------------------------------------------------- gradients ---

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


@pytest.mark.parametrize("T,D,eps,pos0", [(5, 4, 1e-6, 0), (8, 8, 1e-2, 3), (6, 6, 1e-6, 11)])
def test_backward_matches_finite_differences(T, D, eps, pos0):
    B, H = 1, 1
    q, k, v, do = (_rand((B, T, H, D), 40 + s) for s in range(4))
    pos = np.arange(T) + pos0

    def loss(qq, kk, vv):
        o, _ = oracle.attn_fwd(qq, kk, vv, pos=pos, eps=eps)
        return float(np.sum(o * do))

    dq, dk, dv = oracle.attn_bwd(q, k, v, do, pos=pos, eps=eps)
    for mine, fd in ((dq, _fd_grad(lambda x: loss(x, k, v), q)),
                     (dk, _fd_grad(lambda x: loss(q, x, v), k)),
                     (dv, _fd_grad(lambda x: loss(q, k, x), v))):
        rel = np.linalg.norm(mine - fd) / np.linalg.norm(fd)
        assert rel < 1e-6, rel


def test_gradient_invariants():
    """sum_j dv_j = sum_i do_i (rows of P sum to 1); with eps = 0 the loss is
    invariant to rescaling q_t and k_t, so <dq_t, q_t> = <dk_t, k_t> = 0."""
    B, T, H, D = 2, 33, 2, 16
    q, k, v, do = (_rand((B, T, H, D), 50 + s) for s in range(4))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, eps=0.0)
    assert np.allclose(dv.sum(axis=1), do.sum(axis=1), atol=1e-11)
    assert np.max(np.abs(np.sum(dq * q, -1))) < 1e-11
    assert np.max(np.abs(np.sum(dk * k, -1))) < 1e-11


# ----------------------------------------------------------------- decode ---

def test_decode_equals_last_row_of_forward():
    """Decoding the token at position L-1 over cache slots 0..L-1 is row L-1 of
    the forward over that prefix (same raw keys and values)."""
    lens, q, k_raw, v = decode_inputs(B=4, H=3, D=32, Tcap=40, seed=60, lens=[1, 17, 40, 25])
    out = oracle.attn_decode(q, k_raw, v, lens)
    for b, L in enumerate(lens.tolist()):
        qf = k_raw[b:b + 1, :L].clone()  # any query rows before L-1 are irrelevant
        qf[0, L - 1] = q[b]
        o, _ = oracle.attn_fwd(qf, k_raw[b:b + 1, :L], v[b:b + 1, :L])
        assert np.allclose(out[b], o[0, L - 1], atol=1e-13)


def test_decode_single_slot_returns_v():
    lens, q, k_raw, v = decode_inputs(B=2, H=2, D=16, Tcap=8, seed=61, lens=[1, 1])
    out = oracle.attn_decode(q, k_raw, v, lens)
    assert np.array_equal(out, v[:, 0].double().numpy())


def test_inputs_are_seeded_and_bf16():
    a = attn_inputs(1, 8, 2, 16, seed=0)
    b = attn_inputs(1, 8, 2, 16, seed=0)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and torch.equal(x, y)
