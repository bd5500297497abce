"""GPU parity of the FP8 forward (nc_attn_fwd_fp8) against the oracle's FP8
forward (oracle.attn_fwd_fp8: the same E4M3 quantisation of qhat, khat, v
and P, then exact arithmetic), through the C ABI on the same seeded inputs.

Bounds: the forward's (output max-abs 1e-2, relative Frobenius 5e-3, lse
max-abs 1e-2) against the quantised oracle: with the quantisation itself on
both sides, what remains is fp32 against fp64 arithmetic, the bf16 rounding
of the output, and the rare E4M3 rounding decision that the two sides take
differently because their inputs to it differ in the last fp32 bits.  Against
the exact (unquantised) oracle the output must stay within 5% relative
Frobenius, the size of the quantisation error itself (E4M3 carries 3
mantissa bits).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import attn_inputs

pytestmark = pytest.mark.gpu

FWD_MAX_ABS, FWD_REL = 1e-2, 5e-3
EPS, BASE = workloads.EPS, workloads.ROPE_BASE


@pytest.fixture(scope="module")
def nc():
    import causal_attention_rope_nc_b300 as m
    return m


def f64(t):
    return t.detach().double().cpu().numpy()


def rel_frob(a, ref):
    return float(np.linalg.norm(a - ref) / np.linalg.norm(ref))


def run(nc, q, k, v, W=0):
    out, lse = nc.attn_fwd_fp8(q.cuda(), k.cuda(), v.cuda(), eps=EPS, rope_base=BASE, window=W)
    torch.cuda.synchronize()
    assert nc.device_status() == 0
    return f64(out), f64(lse)


def check(o, lse, q, k, v, W=0):
    o_q, lse_q = oracle.attn_fwd_fp8(q, k, v, eps=EPS, base=BASE, window=W)
    assert np.all(np.isfinite(o))
    err = np.max(np.abs(o - o_q))
    assert err <= FWD_MAX_ABS, f"max abs {err}"
    assert rel_frob(o, o_q) <= FWD_REL, f"rel {rel_frob(o, o_q)}"
    assert np.max(np.abs(lse - lse_q)) <= 1e-2
    o_x, _ = oracle.attn_fwd(q, k, v, eps=EPS, base=BASE, window=W)
    assert rel_frob(o, o_x) <= 0.05


@pytest.mark.parametrize("B,T,H,Hkv,W,seed", [
    (1, 256, 2, 2, 0, 401),     # two full query tiles
    (2, 300, 3, 3, 0, 402),     # ragged tail, odd head count
    (1, 1, 2, 2, 0, 403),       # a single token
    (1, 384, 4, 2, 0, 404),     # grouped-query, three tiles (one pair and a lone tile)
    (1, 640, 2, 1, 100, 405),   # multi-query with a window cut inside a tile
    (2, 129, 2, 2, 1, 406),     # window 1: the output is the rounded v
])
def test_fp8_matches_quantised_oracle(nc, B, T, H, Hkv, W, seed):
    q, k, v, _ = attn_inputs(B, T, H, 128, seed, with_dout=False, kv_heads=Hkv)
    o, lse = run(nc, q, k, v, W)
    check(o, lse, q, k, v, W)


def test_fp8_rejects_head_dim_64(nc):
    q, k, v, _ = attn_inputs(1, 64, 1, 64, 407, with_dout=False)
    with pytest.raises(nc.NcError):
        nc.attn_fwd_fp8(q.cuda(), k.cuda(), v.cuda())


def test_fp8_full_size_sampled(nc):
    """The d20 shape at full size in the bench's launch configuration; the
    oracle recomputes three whole (b, h) slices."""
    w = workloads.D20
    q, k, v, _ = workloads.workload_inputs(w, with_dout=False)
    o, lse = run(nc, q, k, v)
    for b, h in ((0, 0), (w.B - 1, w.H - 1), (w.B // 2, w.H // 2)):
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        check(o[sl], lse[b:b + 1, h:h + 1], q[sl].contiguous(), k[sl].contiguous(), v[sl].contiguous())
    assert np.all(np.isfinite(o))
