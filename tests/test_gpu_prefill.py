"""GPU parity of nc_attn_prefill (a chunk of new tokens per stream appended
to a KV cache at a per-stream offset) against the fp64 oracle, with the
forward's tolerances; the cache slots the call writes are checked too, and a
decode step run on the cache it leaves behind."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import prefill_inputs

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


def _prefill(nc, start, q, k_raw, v, W=0):
    """Cache slots before each chunk hold the stream's history (normalised and
    rotated by the library's own prologue); the chunk's slots are zeroed so
    the test sees the call write them."""
    B, C, H, D = q.shape
    kcache = nc.qk_norm_rope(k_raw.cuda(), eps=EPS, rope_base=BASE)
    vcache = v.cuda().clone()
    kc, vc = [], []
    for b, s in enumerate(start.tolist()):
        kc.append(k_raw[b, s:s + C])
        vc.append(v[b, s:s + C])
        kcache[b, s:s + C] = 0
        vcache[b, s:s + C] = 0
    k_chunk = torch.stack(kc).contiguous().cuda()
    v_chunk = torch.stack(vc).contiguous().cuda()
    out, lse = nc.attn_prefill(q.cuda(), k_chunk, v_chunk, start.cuda(), kcache, vcache, eps=EPS, rope_base=BASE,
                               window=W)
    torch.cuda.synchronize()
    assert nc.device_status() == 0
    return out, lse, kcache, vcache


@pytest.mark.parametrize("B,C,H,D,Tcap,start,W,seed", [
    (3, 200, 4, 128, 700, [0, 123, 500], 0, 90),   # two query tiles, ragged; offsets off tile edges
    (2, 300, 2, 64, 900, [256, 600], 100, 91),      # D = 64, window cut inside a tile, 3 query tiles
    (2, 1, 3, 128, 64, [0, 63], 0, 92),             # single-token chunks (a decode through this path)
    (1, 128, 2, 128, 2048, [1920], 512, 93),        # one full tile at the end of a long cache, window
])
def test_prefill_matches_oracle(nc, B, C, H, D, Tcap, start, W, seed):
    start_t, q, k_raw, v = prefill_inputs(B, C, H, D, Tcap, seed, start=start)
    out, lse, kcache, vcache = _prefill(nc, start_t, q, k_raw, v, W)
    o_ref, lse_ref = oracle.attn_prefill(q, k_raw, v, start_t, eps=EPS, base=BASE, window=W)
    o = f64(out)
    assert np.max(np.abs(o - o_ref)) <= FWD_MAX_ABS
    assert rel_frob(o, o_ref) <= FWD_REL
    assert np.max(np.abs(f64(lse) - lse_ref)) <= 1e-2
    # the chunk's keys (normalised, rotated at their positions, rounded to the
    # bf16 cache: half a bf16 ulp, 2^-8 relative) and values are in the cache
    kc, vc = kcache.cpu(), vcache.cpu()
    for b, s in enumerate(start):
        kr, _ = oracle.norm_rope(k_raw[b:b + 1, s:s + C], pos=list(range(s, s + C)), eps=EPS, base=BASE)
        got = f64(kc[b, s:s + C])
        assert np.all(np.abs(got - kr[0]) <= np.abs(kr[0]) * 2.0 ** -8 + 1e-4)
        assert torch.equal(vc[b, s:s + C], v[b, s:s + C])


def test_two_chunks_equal_one_forward(nc):
    """A prompt fed in two chunks gives the rows of one forward over the whole
    prompt: both chunks' outputs against the oracle's forward, at the
    forward's tolerances."""
    B, H, D, T, a = 2, 3, 128, 333, 150
    start_t, q, k_raw, v = prefill_inputs(B, T, H, D, T, seed=94, start=[0, 0])
    o_ref, _ = oracle.attn_fwd(q, k_raw, v, eps=EPS, base=BASE)
    kcache = torch.zeros((B, T, H, D), dtype=torch.bfloat16, device="cuda")
    vcache = torch.zeros((B, T, H, D), dtype=torch.bfloat16, device="cuda")
    o1, _ = nc.attn_prefill(q[:, :a].contiguous().cuda(), k_raw[:, :a].contiguous().cuda(),
                            v[:, :a].contiguous().cuda(), torch.zeros(B, dtype=torch.int32, device="cuda"),
                            kcache, vcache, eps=EPS, rope_base=BASE)
    o2, _ = nc.attn_prefill(q[:, a:].contiguous().cuda(), k_raw[:, a:].contiguous().cuda(),
                            v[:, a:].contiguous().cuda(), torch.full((B,), a, dtype=torch.int32, device="cuda"),
                            kcache, vcache, eps=EPS, rope_base=BASE)
    torch.cuda.synchronize()
    assert nc.device_status() == 0
    both = f64(torch.cat([o1, o2], dim=1))
    assert np.max(np.abs(both - o_ref)) <= FWD_MAX_ABS
    assert rel_frob(both, o_ref) <= FWD_REL


def test_decode_after_prefill(nc):
    """Prefill a prompt, then decode the next token on the cache it wrote."""
    B, H, D, Tcap, C = 2, 4, 128, 512, 300
    start_t, q, k_raw, v = prefill_inputs(B, C, H, D, Tcap, seed=95, start=[0, 100])
    kcache = torch.zeros((B, Tcap, H, D), dtype=torch.bfloat16, device="cuda")
    vcache = torch.zeros((B, Tcap, H, D), dtype=torch.bfloat16, device="cuda")
    # history before the chunk of stream 1 through the library's prologue
    kcache[1, :100] = nc.qk_norm_rope(k_raw[1:2, :100].contiguous().cuda(), eps=EPS, rope_base=BASE)[0]
    vcache[1, :100] = v[1, :100].cuda()
    kc = torch.stack([k_raw[b, s:s + C] for b, s in enumerate(start_t.tolist())]).contiguous().cuda()
    vc = torch.stack([v[b, s:s + C] for b, s in enumerate(start_t.tolist())]).contiguous().cuda()
    nc.attn_prefill(q.cuda(), kc, vc, start_t.cuda(), kcache, vcache, eps=EPS, rope_base=BASE)
    lens = start_t + C + 1
    qn = workloads.randn_bf16((B, H, D), torch.Generator().manual_seed(96))
    k_new = torch.stack([k_raw[b, L - 1] for b, L in enumerate(lens.tolist())]).contiguous()
    v_new = torch.stack([v[b, L - 1] for b, L in enumerate(lens.tolist())]).contiguous()
    out = nc.attn_decode(qn.cuda(), kcache, vcache, lens.cuda(), k_new=k_new.cuda(), v_new=v_new.cuda(),
                         eps=EPS, rope_base=BASE)
    torch.cuda.synchronize()
    assert nc.device_status() == 0
    ref = oracle.attn_decode(qn, k_raw, v, lens, eps=EPS, base=BASE)
    assert np.max(np.abs(f64(out) - ref)) <= FWD_MAX_ABS
