"""The bounds-checked debug build (libncattn_check.so, compiled with
-DNC_CHECK) on the small and edge cases, as a stand-in for a memory checker.

In that build every raw global store and the decode kernels' raw cache loads
are checked against the tensors the call registered (its outputs and
workspace for stores, all of its tensors for loads); a stray access is
skipped and recorded in the library's status word.  TMA copies are clipped
to their tensors by the tensor maps.  Here, in addition, every output and
workspace is allocated inside a larger buffer whose bands before and after
it hold a canary pattern.

Each case checks that:
  - the checked build's status word stays 0 (no access left its tensor);
  - every guard band still holds the canary;
  - the outputs are bit-identical to the normal build's on the same inputs.
"""
import ctypes

import pytest
import torch

import workloads
from workloads import attn_inputs, decode_inputs, prefill_inputs

pytestmark = pytest.mark.gpu

EPS, BASE = workloads.EPS, workloads.ROPE_BASE
GUARD_BYTES = 8192  # canary band on each side of every output


@pytest.fixture(scope="module")
def libs():
    import causal_attention_rope_nc_b300 as nc
    return nc, nc._load(nc.LIB_CHECK_PATH)


CANARY = {torch.bfloat16: 0x7BAD, torch.float16: 0x7BAD, torch.float32: 0x7FBADBAD, torch.uint8: 0xA5,
          torch.int32: 0x5A5A5A5A}
INT_VIEW = {torch.bfloat16: torch.int16, torch.float16: torch.int16, torch.float32: torch.int32,
            torch.uint8: torch.uint8, torch.int32: torch.int32}


class Guarded:
    """A tensor inside a buffer with canary bands of GUARD_BYTES on both sides."""

    def __init__(self, shape, dtype, init=None):
        esz = torch.empty((), dtype=dtype).element_size()
        self.g = GUARD_BYTES // esz
        n = 1
        for s in shape:
            n *= s
        self.n = n
        self.buf = torch.empty(n + 2 * self.g, dtype=dtype, device="cuda")
        iv = self.buf.view(INT_VIEW[dtype])
        c = CANARY[dtype]
        if INT_VIEW[dtype] == torch.int16 and c >= 1 << 15:
            c -= 1 << 16
        iv.fill_(c)
        self.canary = c
        self.t = self.buf[self.g:self.g + n].view(shape)
        if init is not None:
            self.t.copy_(init)

    def intact(self):
        iv = self.buf.view(INT_VIEW[self.buf.dtype])
        return bool((iv[: self.g] == self.canary).all()) and bool((iv[self.g + self.n:] == self.canary).all())


def P(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def status(chk):
    st = ctypes.c_uint(0)
    assert chk.nc_device_status(None, ctypes.byref(st)) == 0
    return st.value


def ok(rc, chk):
    assert rc == 0, chk.nc_strerror(rc)


def ws_guarded(nc, op, B, T, H, D):
    n = max(nc.workspace_size(op, B, T, H, D), 1)
    return Guarded((n,), torch.uint8, torch.zeros(n, dtype=torch.uint8, device="cuda"))


@pytest.mark.parametrize("B,T,H,Hkv,D,W", [
    (1, 1, 2, 2, 128, 0),
    (2, 129, 2, 2, 128, 0),
    (1, 257, 2, 1, 64, 0),
    (1, 300, 3, 3, 128, 100),
])
def test_checked_fwd_bwd(libs, B, T, H, Hkv, D, W):
    nc, chk = libs
    q, k, v, dout = (x.cuda() for x in attn_inputs(B, T, H, D, 700 + T, kv_heads=Hkv))
    stream = torch.cuda.current_stream().cuda_stream
    # the normal build's results
    o_ref, lse_ref, qh_ref, kh_ref = nc.attn_fwd(q, k, v, eps=EPS, rope_base=BASE, window=W)
    g_ref = nc.attn_bwd(q, k, v, o_ref, lse_ref, qh_ref, kh_ref, dout, eps=EPS, rope_base=BASE, window=W)
    # the checked build's, every output and workspace inside canary bands
    out = Guarded(q.shape, torch.bfloat16)
    lse = Guarded((B, H, T), torch.float32)
    qh, kh = Guarded(q.shape, torch.float16), Guarded(k.shape, torch.float16)
    wf = ws_guarded(nc, nc.NC_OP_FWD, B, T, H, D)
    ok(chk.nc_attn_fwd_ex(P(q), P(k), P(v), None, P(out.t), P(lse.t), P(qh.t), P(kh.t), None, P(wf.t), wf.n,
                          B, T, H, D, EPS, BASE, W, Hkv, stream), chk)
    dq, dk, dv = Guarded(q.shape, torch.bfloat16), Guarded(k.shape, torch.bfloat16), Guarded(v.shape, torch.bfloat16)
    wb = ws_guarded(nc, nc.NC_OP_BWD, B, T, H, D)
    ok(chk.nc_attn_bwd_ex(P(q), P(k), P(v), None, P(out.t), P(lse.t), P(qh.t), P(kh.t), P(dout), P(dq.t), P(dk.t),
                          P(dv.t), P(wb.t), wb.n, B, T, H, D, EPS, BASE, W, Hkv, stream), chk)
    torch.cuda.synchronize()
    assert status(chk) == 0
    for g in (out, lse, qh, kh, wf, dq, dk, dv, wb):
        assert g.intact()
    assert torch.equal(out.t, o_ref) and torch.equal(lse.t, lse_ref)
    assert torch.equal(qh.t, qh_ref) and torch.equal(kh.t, kh_ref)
    for got, ref in zip((dq.t, dk.t, dv.t), g_ref):
        assert torch.equal(got, ref)


@pytest.mark.parametrize("lens,Hkv", [([1, 256], 4), ([256, 1, 200], 2)])
def test_checked_decode(libs, lens, Hkv):
    """Decode at lengths 1 and Tcap (the new token in the first and in the
    last slot), multi-head (the register kernel) and grouped-query (the TMA
    ring kernel)."""
    nc, chk = libs
    H, D, Tcap = 4, 128, 256
    B = len(lens)
    lens_t, q, k_raw, v = decode_inputs(B, H, D, Tcap, 710, lens=lens, kv_heads=Hkv)
    idx = (lens_t - 1).long()
    k_new = k_raw[torch.arange(B), idx].contiguous().cuda()
    v_new = v[torch.arange(B), idx].contiguous().cuda()
    kc0 = nc.qk_norm_rope(k_raw.cuda(), eps=EPS, rope_base=BASE)
    vc0 = v.cuda()
    qd, ld = q.cuda(), lens_t.cuda()
    ref = nc.attn_decode(qd, kc0.clone(), vc0.clone(), ld, k_new=k_new, v_new=v_new, eps=EPS, rope_base=BASE)
    kc, vc = Guarded(kc0.shape, torch.bfloat16, kc0), Guarded(vc0.shape, torch.bfloat16, vc0)
    out = Guarded((B, H, D), torch.bfloat16)
    ws = ws_guarded(nc, nc.NC_OP_DECODE, B, Tcap, H, D)
    ok(chk.nc_attn_decode_ex(P(qd), P(k_new), P(v_new), P(kc.t), P(vc.t), P(ld), P(out.t), P(ws.t), ws.n, B, H, D,
                             Tcap, EPS, BASE, 0, Hkv, torch.cuda.current_stream().cuda_stream), chk)
    torch.cuda.synchronize()
    assert status(chk) == 0
    for g in (kc, vc, out, ws):
        assert g.intact()
    assert torch.equal(out.t, ref)


def test_checked_prefill_at_cache_end(libs):
    """A chunk that ends exactly at the last cache slot."""
    nc, chk = libs
    B, C, H, D, Tcap = 2, 100, 2, 128, 300
    start = [Tcap - C, Tcap - C]
    start_t, q, k_raw, v = prefill_inputs(B, C, H, D, Tcap, 720, start=start)
    kc0 = nc.qk_norm_rope(k_raw.cuda(), eps=EPS, rope_base=BASE)
    vc0 = v.cuda()
    qd = q.cuda()
    kcn = k_raw[:, Tcap - C:].contiguous().cuda()
    vcn = v[:, Tcap - C:].contiguous().cuda()
    st = start_t.cuda()
    kr, vr = kc0.clone(), vc0.clone()
    o_ref, l_ref = nc.attn_prefill(qd, kcn, vcn, st, kr, vr, eps=EPS, rope_base=BASE)
    kc, vc = Guarded(kc0.shape, torch.bfloat16, kc0), Guarded(vc0.shape, torch.bfloat16, vc0)
    out, lse = Guarded(qd.shape, torch.bfloat16), Guarded((B, H, C), torch.float32)
    ws = ws_guarded(nc, nc.NC_OP_PREFILL, B, C, H, D)
    ok(chk.nc_attn_prefill(P(qd), P(kcn), P(vcn), P(st), P(kc.t), P(vc.t), P(out.t), P(lse.t), P(ws.t), ws.n, B, C,
                           H, D, Tcap, EPS, BASE, 0, H, torch.cuda.current_stream().cuda_stream), chk)
    torch.cuda.synchronize()
    assert status(chk) == 0
    for g in (kc, vc, out, lse, ws):
        assert g.intact()
    assert torch.equal(out.t, o_ref) and torch.equal(lse.t, l_ref)
    assert torch.equal(kc.t, kr) and torch.equal(vc.t, vr)


def test_checked_fp8_forward(libs):
    nc, chk = libs
    B, T, H, D = 1, 300, 2, 128
    q, k, v, _ = (x.cuda() if x is not None else None for x in attn_inputs(B, T, H, D, 730, with_dout=False))
    o_ref, l_ref = nc.attn_fwd_fp8(q, k, v, eps=EPS, rope_base=BASE)
    out, lse = Guarded(q.shape, torch.bfloat16), Guarded((B, H, T), torch.float32)
    ws = ws_guarded(nc, nc.NC_OP_FWD_FP8, B, T, H, D)
    ok(chk.nc_attn_fwd_fp8(P(q), P(k), P(v), None, P(out.t), P(lse.t), P(ws.t), ws.n, B, T, H, D, EPS, BASE, 0, H,
                           torch.cuda.current_stream().cuda_stream), chk)
    torch.cuda.synchronize()
    assert status(chk) == 0
    for g in (out, lse, ws):
        assert g.intact()
    assert torch.equal(out.t, o_ref) and torch.equal(lse.t, l_ref)
