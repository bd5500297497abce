"""Full-size checks on EVERY (b, h) slice and row of the d20 fwd+bwd, from
identities of the method itself (no oracle call), so that no tile of the
grid -- whichever CTA took it from the work counters -- escapes a check:

- softmax rows sum to one, so the key-side gradient sums to the query-side
  one: sum_j dv_j = sum_i dout_i per (batch, key/value head), over the G
  query heads of the group (nanochat page, "Карта репозитория": the GPT
  block's attention; any mask keeps the identity, since every query sees at
  least its own key);
- the RMSNorm has no gain, so the gradient with respect to a raw row is
  orthogonal to that row up to eps / (mean(x^2) + eps):
  <dq_i, q_i> = <dk_j, k_j> = 0 for every row;
- the diagonal score is inside the softmax denominator and every score is
  bounded by |qhat| |khat| / sqrt(D) = sqrt(D):
  qhat_i . khat_i / sqrt(D) <= lse_i <= sqrt(D) + ln(i + 1);
- an output row is a convex combination of the visible value rows, so each
  component lies between the running minimum and maximum of v over keys
  0..i (the window only shrinks that set).
"""
import math

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

EPS, BASE = workloads.EPS, workloads.ROPE_BASE


@pytest.fixture(scope="module")
def nc():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import causal_attention_rope_nc_b300 as m
    return m


@pytest.mark.parametrize("window,kv_heads", [(0, None), (512, None), (0, 2), (512, 2)])
def test_d20_invariants_every_slice(nc, window, kv_heads):
    w = workloads.D20
    q, k, v, dout = workloads.workload_inputs(w)
    if kv_heads:
        k, v = k[:, :, :kv_heads].contiguous(), v[:, :, :kv_heads].contiguous()
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, dout))
    out, lse, qh, kh = nc.attn_fwd(qd, kd, vd, eps=EPS, rope_base=BASE, window=window)
    dq, dk, dv = nc.attn_bwd(qd, kd, vd, out, lse, qh, kh, dod, eps=EPS, rope_base=BASE, window=window)
    torch.cuda.synchronize()
    assert nc.device_status() == 0
    B, T, H, D = q.shape
    Hkv = k.shape[2]
    G = H // Hkv
    for t in (out, lse, dq, dk, dv):
        assert bool(torch.isfinite(t.float()).all())

    # sum over keys of dv = sum over the group's queries of dout, per (b, kv head)
    sdv = dv.double().sum(1)                                  # [B, Hkv, D]
    sdo = dod.double().sum(1).view(B, Hkv, G, D).sum(2)       # [B, Hkv, D]
    err = (sdv - sdo).norm(dim=-1) / sdo.norm(dim=-1)
    assert float(err.max()) <= 2e-2, f"sum dv vs sum dout: worst slice {float(err.max())}"

    # gradients orthogonal to their raw rows
    for name, g, x in (("dq", dq, qd), ("dk", dk, kd)):
        g64, x64 = g.double(), x.double()
        cos = (g64 * x64).sum(-1).abs() / (g64.norm(dim=-1) * x64.norm(dim=-1) + 1e-300)
        assert float(cos.max()) <= 1e-2, f"{name} not orthogonal to its row: worst {float(cos.max())}"

    # lse between the diagonal score and sqrt(D) + ln(visible keys)
    kh_q = kh.repeat_interleave(G, dim=2) if G > 1 else kh   # key head of each query head
    diag = (qh.double() * kh_q.double()).sum(-1) / math.sqrt(D)  # [B, T, H]
    lse_t = lse.double().permute(0, 2, 1)                       # [B, T, H]
    assert float((diag - lse_t).max()) <= 1e-2, "lse below the diagonal score"
    n_vis = torch.arange(1, T + 1, device="cuda", dtype=torch.float64)
    if window:
        n_vis = n_vis.clamp(max=window)
    upper = math.sqrt(D) + torch.log(n_vis)[None, :, None]
    assert float((lse_t - upper).max()) <= 1e-2, "lse above sqrt(D) + ln(visible keys)"

    # out inside the running hull of v over keys 0..i
    v_q = vd.repeat_interleave(G, dim=2) if G > 1 else vd
    vmax = torch.cummax(v_q.float(), dim=1).values
    vmin = torch.cummin(v_q.float(), dim=1).values
    o = out.float()
    slack = 1e-2 * (1 + vmax.abs())
    assert bool((o <= vmax + slack).all()) and bool((o >= vmin - slack).all()), "out outside the hull of v"
