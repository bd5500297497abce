"""GPU parity of grouped-query attention (Hkv key/value heads shared by groups
of H / Hkv consecutive query heads) through nc_attn_fwd_ex, nc_attn_bwd_ex,
nc_attn_decode_ex and nc_attn_prefill, against the fp64 oracle on the same
seeded bf16 inputs, with the tolerances of tests/test_gpu_parity.py.  Group
sizes 2, 3 and H (one key/value head: multi-query attention) are covered, with
and without a sliding window, ragged sequence tails and D = 64 and 128."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import attn_inputs, decode_inputs, prefill_inputs

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


def bf16_close(got, ref):
    """A bf16 rounding of ref (at most half a bf16 ulp, 2^-8 relative), up to
    the fp32 arithmetic before it."""
    return bool(np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-3))


def run(nc, q, k, v, dout, W=0):
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, dout))
    out, lse, qh, kh = nc.attn_fwd(qd, kd, vd, eps=EPS, rope_base=BASE, window=W)
    dq, dk, dv = nc.attn_bwd(qd, kd, vd, out, lse, qh, kh, dod, eps=EPS, rope_base=BASE, window=W)
    torch.cuda.synchronize()
    assert nc.device_status() == 0
    return out, lse, qh, kh, dq, dk, dv


@pytest.mark.parametrize("B,T,H,Hkv,D,W,seed", [
    (1, 300, 4, 2, 128, 0, 101),    # pairs of query heads, ragged tail
    (2, 640, 6, 2, 64, 0, 102),     # groups of 3, D = 64
    (1, 385, 4, 1, 128, 129, 103),  # one key/value head (multi-query), window edge inside a tile
    (2, 256, 8, 4, 128, 0, 104),    # two full tiles
    (1, 1000, 6, 3, 128, 250, 105), # window not a multiple of the tile, several tiles per group
    (1, 1, 4, 1, 128, 0, 110),      # single token, one key/value head
    (2, 128, 4, 2, 64, 0, 111),     # exactly one tile per head
])
def test_gqa_fwd_bwd_matches_oracle(nc, B, T, H, Hkv, D, W, seed):
    q, k, v, dout = attn_inputs(B, T, H, D, seed, kv_heads=Hkv)
    out, lse, _, kh, dq, dk, dv = run(nc, q, k, v, dout, W)
    assert tuple(kh.shape) == (B, T, Hkv, D) and tuple(dk.shape) == (B, T, Hkv, D)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, eps=EPS, base=BASE, window=W)
    o = f64(out)
    assert np.max(np.abs(o - o_ref)) <= FWD_MAX_ABS
    assert rel_frob(o, o_ref) <= FWD_REL
    assert np.max(np.abs(f64(lse) - lse_ref)) <= 1e-2
    g_ref = oracle.attn_bwd(q, k, v, dout, eps=EPS, base=BASE, window=W)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), g_ref):
        assert rel_frob(f64(got), ref) <= GRAD_REL, name


def test_gqa_forward_is_mha_on_repeated_heads(nc):
    """Every query head reads its group's key/value tiles, so the forward (out,
    lse, qhat) is bit-identical to the multi-head call on key/value heads
    repeated per group, and khat is the repeated call's first head of each
    group; dq matches too.  dk and dv of the grouped call are the group sums
    (accumulated in fp32 before the one bf16 rounding), checked against the
    oracle above."""
    B, T, H, Hkv, D = 2, 333, 6, 2, 128
    G = H // Hkv
    q, k, v, dout = attn_inputs(B, T, H, D, 106, kv_heads=Hkv)
    a = run(nc, q, k, v, dout)
    b = run(nc, q, k.repeat_interleave(G, dim=2), v.repeat_interleave(G, dim=2), dout)
    for x, y in zip(a[:3], b[:3]):  # out, lse, qhat
        assert torch.equal(x, y)
    assert torch.equal(a[3], b[3][:, :, ::G])
    # dq: the same products in the same order, whatever k's head count
    assert torch.equal(a[4], b[4])


def test_gqa_full_size_sampled(nc):
    """The d20 shape with 2 key/value heads of 5 query heads each, at full
    size; the oracle recomputes whole (batch, group) slices."""
    w = workloads.D20
    Hkv = 2
    G = w.H // Hkv
    q, k, v, dout = attn_inputs(w.B, w.T, w.H, w.D, w.seed, kv_heads=Hkv)
    out, _, _, _, dq, dk, dv = run(nc, q, k, v, dout)
    for b, hk in [(0, 0), (w.B - 1, Hkv - 1)]:
        qs = (slice(b, b + 1), slice(None), slice(hk * G, hk * G + G))
        ks = (slice(b, b + 1), slice(None), slice(hk, hk + 1))
        o_ref, _ = oracle.attn_fwd(q[qs], k[ks], v[ks], eps=EPS, base=BASE)
        o = f64(out[qs])
        assert np.max(np.abs(o - o_ref)) <= FWD_MAX_ABS
        assert rel_frob(o, o_ref) <= FWD_REL
        g_ref = oracle.attn_bwd(q[qs], k[ks], v[ks], dout[qs], eps=EPS, base=BASE)
        for got, sl, ref in zip((dq, dk, dv), (qs, ks, ks), g_ref):
            assert rel_frob(f64(got[sl]), ref) <= GRAD_REL


@pytest.mark.parametrize("H,Hkv,D,lens,W,new", [
    (8, 2, 128, [1, 2048, 777, 300], 0, False),
    (12, 4, 128, [129, 1, 2048, 1000], 0, True),   # the new token written once per key/value head
    (16, 1, 64, [64, 65, 2000, 513], 0, True),     # multi-query, D = 64
    (10, 5, 128, [2048, 1, 1000, 513], 300, True), # window
    (32, 8, 128, [2048, 700, 1, 129], 0, True),    # 32 query heads: two per compute warp
    (48, 16, 64, [1500, 2048, 64, 2], 0, True),    # 48 query heads: four per compute warp
    (32, 16, 128, [2048, 333, 1, 130], 0, True),   # 64 KB stages: a ring of one stage
])
def test_gqa_decode_matches_oracle(nc, H, Hkv, D, lens, W, new):
    Tcap = 2048
    lens_t, q, k_raw, v = decode_inputs(B=len(lens), H=H, D=D, Tcap=Tcap, seed=107, lens=lens, kv_heads=Hkv)
    kcache = nc.qk_norm_rope(k_raw.cuda(), eps=EPS, rope_base=BASE)
    vcache = v.cuda().clone()
    k_new = v_new = None
    if new:  # the new token's slot starts empty: the call must fill it
        idx = (torch.arange(len(lens)), lens_t.long() - 1)
        k_new = k_raw[idx].contiguous().cuda()
        v_new = v[idx].contiguous().cuda()
        idx_d = tuple(i.cuda() for i in idx)
        kcache[idx_d] = 0
        vcache[idx_d] = 0
    out = nc.attn_decode(q.cuda(), kcache, vcache, lens_t.cuda(), k_new=k_new, v_new=v_new, eps=EPS,
                         rope_base=BASE, window=W)
    torch.cuda.synchronize()
    assert nc.device_status() == 0
    assert tuple(out.shape) == (len(lens), H, D)
    ref = oracle.attn_decode(q, k_raw, v, lens_t, eps=EPS, base=BASE, window=W)
    o = f64(out)
    assert np.max(np.abs(o - ref)) <= FWD_MAX_ABS
    assert rel_frob(o, ref) <= FWD_REL
    if new:  # every key/value head of the new slot: normalised, rotated at its position (bf16), and v
        kc, vc = kcache.cpu(), vcache.cpu()
        for b, L in enumerate(lens):
            kr, _ = oracle.norm_rope(k_raw[b:b + 1, L - 1:L], pos=[L - 1], eps=EPS, base=BASE)
            assert bf16_close(f64(kc[b, L - 1]), kr[0, 0])
            assert torch.equal(vc[b, L - 1], v[b, L - 1])


@pytest.mark.parametrize("B,C,H,Hkv,D,Tcap,start,W,seed", [
    (3, 200, 4, 2, 128, 700, [0, 123, 500], 0, 108),
    (2, 300, 6, 1, 64, 900, [256, 600], 100, 109),
])
def test_gqa_prefill_matches_oracle(nc, B, C, H, Hkv, D, Tcap, start, W, seed):
    start_t, q, k_raw, v = prefill_inputs(B, C, H, D, Tcap, seed, start=start, kv_heads=Hkv)
    kcache = nc.qk_norm_rope(k_raw.cuda(), eps=EPS, rope_base=BASE)
    vcache = v.cuda().clone()
    kc, vc = [], []
    for b, s in enumerate(start):
        kc.append(k_raw[b, s:s + C])
        vc.append(v[b, s:s + C])
        kcache[b, s:s + C] = 0
        vcache[b, s:s + C] = 0
    k_chunk = torch.stack(kc).contiguous().cuda()
    v_chunk = torch.stack(vc).contiguous().cuda()
    out, lse = nc.attn_prefill(q.cuda(), k_chunk, v_chunk, start_t.cuda(), kcache, vcache, eps=EPS,
                               rope_base=BASE, window=W)
    torch.cuda.synchronize()
    assert nc.device_status() == 0
    o_ref, lse_ref = oracle.attn_prefill(q, k_raw, v, start_t, eps=EPS, base=BASE, window=W)
    o = f64(out)
    assert np.max(np.abs(o - o_ref)) <= FWD_MAX_ABS
    assert rel_frob(o, o_ref) <= FWD_REL
    assert np.max(np.abs(f64(lse) - lse_ref)) <= 1e-2
    kc, vc = kcache.cpu(), vcache.cpu()
    for b, s in enumerate(start):
        kr, _ = oracle.norm_rope(k_raw[b:b + 1, s:s + C], pos=list(range(s, s + C)), eps=EPS, base=BASE)
        assert bf16_close(f64(kc[b, s:s + C]), kr[0])
        assert torch.equal(vc[b, s:s + C], v[b, s:s + C])
