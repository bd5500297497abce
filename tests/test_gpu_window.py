"""GPU parity of the sliding-window calls (nc_attn_fwd_ex, nc_attn_bwd_ex,
nc_attn_decode_ex) against the fp64 oracle with the same window, on the same
seeded bf16 inputs and with the tolerances of tests/test_gpu_parity.py.
Windows are chosen so that the band edge falls inside a 128-key tile (W not a
multiple of 128), on a tile boundary (W = 512, the quarter of a 2048 context),
and at the degenerate ends (W = 1: every query sees only itself; W >= T: the
plain causal mask, bit-identical to the causal calls)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import attn_inputs, decode_inputs

pytestmark = pytest.mark.gpu

FWD_MAX_ABS, FWD_REL, GRAD_REL = 1e-2, 5e-3, 1e-2
EPS, BASE = workloads.EPS, workloads.ROPE_BASE


@pytest.fixture(scope="module")
def nc():
    import causal_attention_rope_nc_b300 as m
    return m


def f64(t):
    return t.detach().double().cpu().numpy()


def rel_frob(a, ref):
    nr = np.linalg.norm(ref)
    return float(np.linalg.norm(a - ref) / nr) if nr else float(np.max(np.abs(a)))


def run(nc, q, k, v, dout, W):
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, dout))
    out, lse, qh, kh = nc.attn_fwd(qd, kd, vd, eps=EPS, rope_base=BASE, window=W)
    dq, dk, dv = nc.attn_bwd(qd, kd, vd, out, lse, qh, kh, dod, eps=EPS, rope_base=BASE, window=W)
    torch.cuda.synchronize()
    assert nc.device_status() == 0
    return out, lse, dq, dk, dv


@pytest.mark.parametrize("B,T,H,D,W,seed", [
    (1, 300, 3, 128, 100, 71),   # band edge inside a tile, ragged tail
    (2, 640, 2, 64, 257, 72),    # D = 64, edge one past two tiles
    (1, 2048, 2, 128, 512, 73),  # a quarter of a 2048 context: edge on a tile boundary
    (1, 129, 2, 128, 1, 74),     # every query sees only itself
    (1, 385, 1, 128, 129, 75),   # edge one row into the second tile back
])
def test_window_fwd_bwd_matches_oracle(nc, B, T, H, D, W, seed):
    q, k, v, dout = attn_inputs(B, T, H, D, seed)
    out, lse, dq, dk, dv = run(nc, q, k, v, dout, W)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, eps=EPS, base=BASE, window=W)
    o = f64(out)
    assert np.max(np.abs(o - o_ref)) <= FWD_MAX_ABS
    assert rel_frob(o, o_ref) <= FWD_REL
    assert np.max(np.abs(f64(lse) - lse_ref)) <= 1e-2
    g_ref = oracle.attn_bwd(q, k, v, dout, eps=EPS, base=BASE, window=W)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), g_ref):
        assert rel_frob(f64(got), ref) <= GRAD_REL, name


def test_window_one_gives_v(nc):
    """W = 1: the output is v (rounded to bf16), whatever q and k are."""
    q, k, v, dout = attn_inputs(2, 200, 2, 128, 76)
    out, *_ = run(nc, q, k, v, dout, 1)
    assert torch.equal(out.cpu(), v)


@pytest.mark.parametrize("W", [300, 4096])
def test_window_at_least_T_is_the_causal_call(nc, W):
    """window >= T takes exactly the causal path: bit-identical results."""
    q, k, v, dout = attn_inputs(1, 300, 2, 128, 77)
    a = run(nc, q, k, v, dout, W)
    b = run(nc, q, k, v, dout, 0)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_window_full_size_sampled(nc):
    """The d20 shape with the short-window layers' W = T/4, at full size; the
    oracle recomputes whole (b, h) slices."""
    w = workloads.D20
    W = w.T // 4
    q, k, v, dout = workloads.workload_inputs(w)
    out, lse, dq, dk, dv = run(nc, q, k, v, dout, W)
    for b, h in [(0, 0), (w.B - 1, w.H - 1), (w.B // 2, w.H // 2)]:
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        o_ref, _ = oracle.attn_fwd(q[sl], k[sl], v[sl], eps=EPS, base=BASE, window=W)
        o = f64(out[sl])
        assert np.max(np.abs(o - o_ref)) <= FWD_MAX_ABS
        g_ref = oracle.attn_bwd(q[sl], k[sl], v[sl], dout[sl], eps=EPS, base=BASE, window=W)
        for got, ref in zip((dq, dk, dv), g_ref):
            assert rel_frob(f64(got[sl]), ref) <= GRAD_REL


@pytest.mark.parametrize("lens,W", [([1, 2048, 777, 300], 512), ([64, 65, 129, 2048], 100),
                                    ([2048, 1, 1000, 513], 1)])
def test_window_decode_matches_oracle(nc, lens, W):
    lens_t, q, k_raw, v = decode_inputs(B=len(lens), H=10, D=128, Tcap=2048, seed=78, lens=lens)
    kcache = nc.qk_norm_rope(k_raw.cuda(), eps=EPS, rope_base=BASE)
    vcache = v.cuda()
    out = nc.attn_decode(q.cuda(), kcache, vcache, lens_t.cuda(), eps=EPS, rope_base=BASE, window=W)
    torch.cuda.synchronize()
    assert nc.device_status() == 0
    ref = oracle.attn_decode(q, k_raw, v, lens_t, eps=EPS, base=BASE, window=W)
    o = f64(out)
    assert np.max(np.abs(o - ref)) <= FWD_MAX_ABS
    assert rel_frob(o, ref) <= FWD_REL
