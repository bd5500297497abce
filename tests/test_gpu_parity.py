"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded bf16 inputs.

Tolerances (bf16 inputs, fp32 accumulation):
  forward output  max |gpu - oracle| <= 1e-2 and ||gpu - oracle||_F / ||oracle||_F <= 5e-3
  lse             max |gpu - oracle| <= 1e-2
  gradients       ||gpu - oracle||_F / ||oracle||_F <= 1e-2
Decode uses the forward bounds.
"""
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


def rel_frob(a, ref):
    """Relative Frobenius error; where the exact reference is identically zero
    (e.g. dq and dk of a single token, whose output v does not depend on q or
    k) the relative error is undefined and the absolute max error is returned
    instead, which must then be rounding noise."""
    nr = np.linalg.norm(ref)
    if nr == 0.0:
        return float(np.max(np.abs(a))) if a.size else 0.0
    return float(np.linalg.norm(a - ref) / nr)


def f64(t):
    return t.detach().double().cpu().numpy()


def assert_bf16_close(got, ref):
    """A bf16 store of ref: at most half a bf16 ulp (2^-8 relative) plus fp32 noise."""
    bound = np.abs(ref) * 2.0 ** -8 + 1e-4
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) - bound))


def check_fwd(out, lse, o_ref, lse_ref):
    o = f64(out)
    assert np.all(np.isfinite(o))
    err = np.max(np.abs(o - o_ref))
    assert err <= FWD_MAX_ABS, f"fwd max abs {err}"
    assert rel_frob(o, o_ref) <= FWD_REL, f"fwd rel {rel_frob(o, o_ref)}"
    lerr = np.max(np.abs(f64(lse) - lse_ref))
    assert lerr <= 1e-2, f"lse max abs {lerr}"


def run_fwd_bwd(nc, q, k, v, dout, pos=None):
    dev = "cuda"
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, dout))
    posd = None if pos is None else torch.as_tensor(pos, dtype=torch.int32, device=dev)
    out, lse, qh, kh = nc.attn_fwd(qd, kd, vd, pos=posd, eps=EPS, rope_base=BASE)
    dq, dk, dv = nc.attn_bwd(qd, kd, vd, out, lse, qh, kh, dod, pos=posd, eps=EPS, rope_base=BASE)
    torch.cuda.synchronize()
    assert nc.device_status() == 0
    return out, lse, qh, kh, dq, dk, dv


SMALL = [
    (1, 128, 2, 64, 0),     # the tiny workload
    (2, 300, 3, 128, 11),   # several tiles + ragged tail
    (1, 257, 2, 64, 12),    # one row past a tile
    (1, 1, 1, 128, 13),     # single token
    (3, 129, 1, 128, 14),   # ragged by one
    (1, 640, 13, 128, 15),  # odd head count, five full tiles
]


@pytest.mark.parametrize("B,T,H,D,seed", SMALL)
def test_fwd_bwd_small(nc, B, T, H, D, seed):
    q, k, v, dout = attn_inputs(B, T, H, D, seed)
    out, lse, qh, kh, dq, dk, dv = run_fwd_bwd(nc, q, k, v, dout)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, eps=EPS, base=BASE)
    check_fwd(out, lse, o_ref, lse_ref)
    qh_ref, _ = oracle.norm_rope(q, eps=EPS, base=BASE)
    assert_bf16_close(f64(qh), qh_ref)
    dq_ref, dk_ref, dv_ref = oracle.attn_bwd(q, k, v, dout, eps=EPS, base=BASE)
    for name, g, r in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        e = rel_frob(f64(g), r)
        assert e <= GRAD_REL, f"{name} rel {e}"


def test_position_offset_uses_pos(nc):
    """RoPE with explicit positions: relative-position invariance holds on the
    GPU (shifted positions give the oracle's unshifted answer), and a
    non-uniform position array matches the oracle with the same positions."""
    B, T, H, D = 1, 200, 2, 128
    q, k, v, dout = attn_inputs(B, T, H, D, 21)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, eps=EPS, base=BASE)
    pos = np.arange(T, dtype=np.int32) + 1000
    out, lse, *_ = run_fwd_bwd(nc, q, k, v, dout, pos=pos)
    check_fwd(out, lse, o_ref, lse_ref)
    pos2 = (np.arange(T) * 3 + 7).astype(np.int32)
    out2, lse2, _, _, dq, dk, dv = run_fwd_bwd(nc, q, k, v, dout, pos=pos2)
    o2_ref, l2_ref = oracle.attn_fwd(q, k, v, pos=pos2, eps=EPS, base=BASE)
    check_fwd(out2, lse2, o2_ref, l2_ref)
    g_ref = oracle.attn_bwd(q, k, v, dout, pos=pos2, eps=EPS, base=BASE)
    for g, r in zip((dq, dk, dv), g_ref):
        assert rel_frob(f64(g), r) <= GRAD_REL


def test_causality_bit_exact(nc):
    B, T, H, D, t0 = 1, 384, 2, 128, 150
    q, k, v, _ = attn_inputs(B, T, H, D, 22)
    out1, lse1, *_ = nc.attn_fwd(q.cuda(), k.cuda(), v.cuda(), eps=EPS, rope_base=BASE)
    g = torch.Generator().manual_seed(99)
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    for a in (q2, k2, v2):
        a[:, t0 + 1:] = torch.randn(a[:, t0 + 1:].shape, generator=g).to(torch.bfloat16)
    out2, lse2, *_ = nc.attn_fwd(q2.cuda(), k2.cuda(), v2.cuda(), eps=EPS, rope_base=BASE)
    assert torch.equal(out1[:, : t0 + 1], out2[:, : t0 + 1])
    assert torch.equal(lse1[..., : t0 + 1], lse2[..., : t0 + 1])


def test_softmax_rows_sum_to_one_on_gpu(nc):
    """v = 1 everywhere: every output is exactly sum_j P_ij = 1 (up to bf16)."""
    B, T, H, D = 2, 333, 2, 128
    q, k, _, _ = attn_inputs(B, T, H, D, 23)
    v = torch.ones(B, T, H, D, dtype=torch.bfloat16)
    out, *_ = nc.attn_fwd(q.cuda(), k.cuda(), v.cuda(), eps=EPS, rope_base=BASE)
    assert float((out.float() - 1).abs().max()) <= 8e-3


def test_repeat_calls_identical(nc):
    """Forward is deterministic; the backward's dQ reductions may reorder but
    stay within tolerance of each other."""
    q, k, v, dout = attn_inputs(2, 256, 2, 128, 24)
    a = run_fwd_bwd(nc, q, k, v, dout)
    b = run_fwd_bwd(nc, q, k, v, dout)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(a[5], b[5]) and torch.equal(a[6], b[6])  # dk, dv: no atomics
    assert rel_frob(f64(a[4]), f64(b[4])) < 1e-3


# ----------------------------------------------------------------- decode ---

def _gpu_decode(nc, lens, q, k_raw, v, with_new=True):
    """Prefill the key cache with the library's own norm+RoPE, then decode the
    token at position lens-1 (optionally writing its key/value first)."""
    B, Tcap, H, D = k_raw.shape
    kr = k_raw.cuda()
    kcache = nc.qk_norm_rope(kr, eps=EPS, rope_base=BASE)
    vcache = v.cuda().clone()
    lens_d = lens.cuda()
    k_new = v_new = None
    if with_new:
        idx = (lens - 1).long()
        k_new = k_raw[torch.arange(B), idx].contiguous().cuda()
        v_new = v[torch.arange(B), idx].contiguous().cuda()
        # scribble over the slot so the test sees the kernel write it
        bi, pi = torch.arange(B, device="cuda"), idx.cuda()
        kcache[bi, pi] = 0
        vcache[bi, pi] = 0
    out = nc.attn_decode(q.cuda(), kcache, vcache, lens_d, k_new=k_new, v_new=v_new, eps=EPS,
                         rope_base=BASE)
    torch.cuda.synchronize()
    assert nc.device_status() == 0
    return out, kcache, vcache


@pytest.mark.parametrize("with_new", [True, False])
def test_decode_full_workload(nc, with_new):
    w = workloads.D20_DECODE
    lens, q, k_raw, v = workloads.decode_workload_inputs(w)
    out, kc, vc = _gpu_decode(nc, lens, q, k_raw, v, with_new)
    ref = oracle.attn_decode(q, k_raw, v, lens, eps=EPS, base=BASE)
    o = f64(out)
    assert np.max(np.abs(o - ref)) <= FWD_MAX_ABS
    assert rel_frob(o, ref) <= FWD_REL
    if with_new:  # the new token's key was normalised, rotated at its position and stored
        kc, vc = kc.cpu(), vc.cpu()
        for b, L in enumerate(lens.tolist()):
            p = L - 1
            kb, _ = oracle.norm_rope(k_raw[b:b + 1, p:p + 1], pos=[p], eps=EPS, base=BASE)
            assert_bf16_close(f64(kc[b, p]), kb[0, 0])
            assert torch.equal(vc[b, p], v[b, p])


@pytest.mark.parametrize("lens", [[1, 1, 1], [2048, 2048, 1], [64, 65, 129], [1, 2048, 777]])
def test_decode_edge_lengths(nc, lens):
    lens_t, q, k_raw, v = decode_inputs(B=len(lens), H=10, D=128, Tcap=2048, seed=31, lens=lens)
    out, *_ = _gpu_decode(nc, lens_t, q, k_raw, v, True)
    ref = oracle.attn_decode(q, k_raw, v, lens_t, eps=EPS, base=BASE)
    assert np.max(np.abs(f64(out) - ref)) <= FWD_MAX_ABS


@pytest.mark.parametrize("H,D,with_new", [(24, 128, True), (40, 64, True), (24, 128, False)])
def test_decode_more_heads_than_warps(nc, H, D, with_new):
    """More than 16 heads: the warps of a CTA take a second head each (the
    first batch of a later head is loaded after the earlier head is done)."""
    lens_t, q, k_raw, v = decode_inputs(B=3, H=H, D=D, Tcap=600, seed=34, lens=[600, 1, 257])
    out, kc, vc = _gpu_decode(nc, lens_t, q, k_raw, v, with_new)
    ref = oracle.attn_decode(q, k_raw, v, lens_t, eps=EPS, base=BASE)
    assert np.max(np.abs(f64(out) - ref)) <= FWD_MAX_ABS
    assert rel_frob(f64(out), ref) <= FWD_REL


def test_decode_head_dim_64_and_repeat(nc):
    lens_t, q, k_raw, v = decode_inputs(B=4, H=3, D=64, Tcap=300, seed=32, lens=[300, 1, 150, 64])
    out1, *_ = _gpu_decode(nc, lens_t, q, k_raw, v, True)
    out2, *_ = _gpu_decode(nc, lens_t, q, k_raw, v, True)  # counters were reset by call 1
    ref = oracle.attn_decode(q, k_raw, v, lens_t, eps=EPS, base=BASE)
    assert np.max(np.abs(f64(out1) - ref)) <= FWD_MAX_ABS
    assert torch.equal(out1, out2)


def test_decode_matches_forward_last_row(nc):
    """Decode of token L-1 equals row L-1 of the GPU forward over the prefix."""
    L, H, D = 700, 4, 128
    q, k, v, _ = attn_inputs(1, L, H, D, 33)
    out_f, *_ = nc.attn_fwd(q.cuda(), k.cuda(), v.cuda(), eps=EPS, rope_base=BASE)
    lens = torch.tensor([L], dtype=torch.int32)
    out_d, *_ = _gpu_decode(nc, lens, q[:, L - 1], k, v, True)
    assert float((out_d.float() - out_f[:, L - 1].float()).abs().max()) <= 1e-2


# -------------------------------------------- full-size, sampled (b, h) ------

@pytest.mark.parametrize("name", ["d12", "d20", "d26"])
def test_full_size_sampled(nc, name):
    """The workload at full size in the bench's launch configuration; the oracle
    recomputes a few whole (b, h) slices (each independent of the others)."""
    w = workloads.ATTN_WORKLOADS[name]
    q, k, v, dout = workloads.workload_inputs(w)
    out, lse, qh, kh, dq, dk, dv = run_fwd_bwd(nc, q, k, v, dout)
    picks = [(0, 0), (w.B - 1, w.H - 1), (w.B // 2, w.H // 2)]
    for b, h in picks:
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        qs, ks, vs, ds = (x[sl].contiguous() for x in (q, k, v, dout))
        o_ref, l_ref = oracle.attn_fwd(qs, ks, vs, eps=EPS, base=BASE)
        check_fwd(out[sl], lse[b:b + 1, h:h + 1], o_ref, l_ref)
        g_ref = oracle.attn_bwd(qs, ks, vs, ds, eps=EPS, base=BASE)
        for nm, g, r in (("dq", dq, g_ref[0]), ("dk", dk, g_ref[1]), ("dv", dv, g_ref[2])):
            e = rel_frob(f64(g[sl]), r)
            assert e <= GRAD_REL, f"{name} ({b},{h}) {nm} rel {e}"
    # properties that hold everywhere: finite outputs, softmax normaliser sane
    for t in (out, dq, dk, dv):
        assert bool(torch.isfinite(t.float()).all())


def test_full_size_forward_first_and_last_batch(nc):
    """d20 forward at full size: every head of the first and of the last batch
    element against the oracle.  The grouped CTA order puts the last (b, h)
    pairs into the grid's tail group, whose tiles run at other group
    positions than the sampled slices above."""
    w = workloads.D20
    q, k, v, _ = workloads.workload_inputs(w, with_dout=False)
    out, lse, *_ = nc.attn_fwd(q.cuda(), k.cuda(), v.cuda(), eps=EPS, rope_base=BASE)
    torch.cuda.synchronize()
    assert nc.device_status() == 0
    for b in (0, w.B - 1):
        for h in range(w.H):
            sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
            qs, ks, vs = (x[sl].contiguous() for x in (q, k, v))
            o_ref, l_ref = oracle.attn_fwd(qs, ks, vs, eps=EPS, base=BASE)
            check_fwd(out[sl], lse[b:b + 1, h:h + 1], o_ref, l_ref)
