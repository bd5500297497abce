"""Pins of the oracle's FP8 forward (orc_attn_fwd_fp8, this library's reading
of fp8 attention: E4M3 qhat and khat scaled by 2^5, v scaled per (batch,
key/value head) by the largest power of two keeping it within 448, P =
exp(s - row max) scaled by 2^8; sums and products in fp64).

What pins it, independently of the oracle's own code:
  - the E4M3 rounding against torch's float8_e4m3fn conversion over a dense
    sweep of the representable range (ties, subnormals, the top binade);
  - quantisation off reproduces the plain forward exactly;
  - closed forms: constant v gives o = 1 (to fp64 rounding), one visible key gives the
    E4M3 rounding of v at its head's scale, uniform scores give the mean of
    the rounded values;
  - a two-token example worked by hand on the E4M3 grid;
  - the q/k scale: a one-hot query and key of head dim 128 (the largest
    element QK-norm allows, sqrt(128) = 11.31) must not saturate.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import attn_inputs

EPS, BASE = workloads.EPS, workloads.ROPE_BASE


def test_e4m3_matches_torch_float8():
    # every representable E4M3 value, the midpoints between neighbours (ties)
    # and points a quarter of the way between them, positive and negative
    grid = torch.arange(0, 256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    grid = np.unique(grid[np.isfinite(grid)])
    grid = grid[grid >= 0]
    mids = (grid[1:] + grid[:-1]) / 2
    quarter = grid[:-1] + (grid[1:] - grid[:-1]) / 4
    x = np.concatenate([grid, mids, quarter, np.linspace(0, 448, 20001)])
    x = np.concatenate([x, -x])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3(x)
    assert np.array_equal(got, ref)


def test_e4m3_saturates():
    """Above 448 the reading saturates (torch's conversion does not: it is not
    the reference here)."""
    assert list(oracle.e4m3(np.array([449.0, 464.0, 1e6, -1e6]))) == [448.0, 448.0, 448.0, -448.0]


def test_quantisation_off_is_the_plain_forward():
    q, k, v, _ = attn_inputs(2, 77, 3, 64, 301)
    o0, l0 = oracle.attn_fwd(q, k, v, eps=EPS, base=BASE)
    o1, l1 = oracle.attn_fwd_fp8(q, k, v, eps=EPS, base=BASE, quant=False)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_constant_values_give_exactly_one():
    """v = 1 everywhere: its scale is 2^8 (448 / 1 -> 2^8.8), 256 is exact in
    E4M3, and every row's quantised weights sum to what divides them (up to
    the fp64 rounding of the division and the sum)."""
    q, k, _, _ = attn_inputs(1, 200, 2, 128, 302)
    v = torch.ones(1, 200, 2, 128)
    o, _ = oracle.attn_fwd_fp8(q, k, v, eps=EPS, base=BASE)
    assert np.max(np.abs(o - 1.0)) < 1e-13


def test_single_key_returns_the_rounded_value():
    """T = 1: o = E4M3(v 2^tau) 2^-tau, tau from the head's largest |v|."""
    q, k, v, _ = attn_inputs(1, 1, 3, 128, 303)
    o, _ = oracle.attn_fwd_fp8(q, k, v, eps=EPS, base=BASE)
    for h in range(3):
        vh = v[0, 0, h].double()
        tau = math.floor(math.log2(448.0 / float(vh.abs().max())))
        exp = (vh * 2.0 ** tau).to(torch.float8_e4m3fn).double() / 2.0 ** tau
        assert np.array_equal(o[0, 0, h], exp.numpy())


def test_uniform_scores_average_the_rounded_values():
    """q = 0: every score is 0, every p = 1, P8 = 256 exactly, so row i is the
    mean of the rounded v over its visible keys."""
    B, T, H, D = 1, 50, 1, 64
    _, k, v, _ = attn_inputs(B, T, H, D, 304)
    q = torch.zeros(B, T, H, D)
    o, lse = oracle.attn_fwd_fp8(q, k, v, eps=EPS, base=BASE)
    vh = v[0, :, 0].double()
    tau = math.floor(math.log2(448.0 / float(vh.abs().max())))
    vr = ((vh * 2.0 ** tau).to(torch.float8_e4m3fn).double() / 2.0 ** tau).numpy()
    for i in range(T):
        assert np.allclose(o[0, i, 0], vr[: i + 1].mean(axis=0), rtol=0, atol=1e-12)
        assert abs(lse[0, 0, i] - math.log(i + 1)) < 1e-12


def test_two_tokens_worked_by_hand():
    """D = 4, both tokens at position 0 (no rotation).  k_0 = e0, k_1 = e1:
    RMSNorm gives 2 e0, 2 e1, times 2^5 = 64 (exact).  q_1 = 2 e0 + e1:
    RMSNorm gives (1.7889, 0.8944), times 2^5 = (57.24, 28.62), rounded on
    the E4M3 grid (spacing 4 in [32, 64), 2 in [16, 32)) to (56, 28), i.e.
    (1.75, 0.875).  Scores (/sqrt(4)): s_10 = 1.75, s_11 = 0.875.  p_11 =
    exp(-0.875) = 0.41686; times 2^8 = 106.72, rounded (spacing 8 in
    [64, 128)) to 104, so the weights are 1 and 104/256.  v_0 = (1, 2, 0, 0),
    v_1 = (-1, 0.5, 0, 0): max 2, scale 2^7, all exact."""
    e = torch.eye(4, dtype=torch.float64)
    k = torch.stack([e[0], e[1]]).reshape(1, 2, 1, 4)
    q = torch.stack([e[0], 2 * e[0] + e[1]]).reshape(1, 2, 1, 4)
    v = torch.tensor([[1.0, 2.0, 0.0, 0.0], [-1.0, 0.5, 0.0, 0.0]], dtype=torch.float64).reshape(1, 2, 1, 4)
    o, lse = oracle.attn_fwd_fp8(q, k, v, pos=[0, 0], eps=0.0, base=BASE)
    w1 = 104.0 / 256.0
    exp1 = (np.array([1.0, 2.0, 0, 0]) + w1 * np.array([-1.0, 0.5, 0, 0])) / (1.0 + w1)
    assert np.allclose(o[0, 0, 0], [1.0, 2.0, 0, 0], rtol=0, atol=1e-15)
    assert np.allclose(o[0, 1, 0], exp1, rtol=0, atol=1e-15)
    assert abs(lse[0, 0, 0] - 2.0) < 1e-15                      # 2 e0 . 2 e0 / 2
    assert abs(lse[0, 0, 1] - (1.75 + math.log(1.0 + math.exp(-0.875)))) < 1e-14


def test_one_hot_head_dim_128_does_not_saturate():
    """q = k = e0 at D = 128: qhat = sqrt(128) e0 = 11.31 e0, times 2^5 =
    362.0, which rounds (spacing 32 in [256, 512)) to 352 = 11.0 * 2^5: the
    score is 121 / sqrt(128).  A larger scale would saturate at 448."""
    e0 = torch.zeros(1, 1, 1, 128, dtype=torch.float64)
    e0[..., 0] = 1.0
    v = torch.ones(1, 1, 1, 128, dtype=torch.float64)
    _, lse = oracle.attn_fwd_fp8(e0, e0, v, eps=0.0, base=BASE)
    assert abs(lse[0, 0, 0] - 121.0 / math.sqrt(128.0)) < 1e-13


@pytest.mark.parametrize("W", [0, 40])
def test_fp8_stays_close_to_the_exact_forward(W):
    """Sanity of the reading, not a parity bound: the quantised forward is
    within a few percent of the exact one on random inputs (E4M3 carries 3
    mantissa bits)."""
    q, k, v, _ = attn_inputs(1, 300, 2, 128, 305)
    o0, _ = oracle.attn_fwd(q, k, v, eps=EPS, base=BASE, window=W)
    o1, _ = oracle.attn_fwd_fp8(q, k, v, eps=EPS, base=BASE, window=W)
    rel = np.linalg.norm(o1 - o0) / np.linalg.norm(o0)
    assert rel < 0.05
