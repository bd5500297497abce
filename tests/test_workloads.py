"""The workload table against the shapes the pages print."""
import os

import pytest

import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "depth_shapes.txt")


def _rows():
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield tuple(int(x) for x in line.split())


@pytest.mark.parametrize("depth,width,heads", list(_rows()))
def test_depth_rule_reproduces_printed_table(depth, width, heads):
    assert workloads.depth_to_shape(depth) == (width, heads)


def test_attention_workloads_follow_depth_rule():
    for w in workloads.ATTN_WORKLOADS.values():
        if w.depth is not None:
            assert (w.width, w.H) == workloads.depth_to_shape(w.depth)
            assert w.D == 128 and w.T == 2048


def test_flop_convention():
    # causal forward: 4*B*H*T^2*D/2; fwd+bwd = 3.5x that (= 7*B*H*T^2*D)
    assert workloads.D20.fwd_flops() == pytest.approx(343.597e9, rel=1e-5)
    assert workloads.D20.fwd_bwd_flops() == pytest.approx(1202.59e9, rel=1e-5)
    assert workloads.D12.fwd_bwd_flops() == pytest.approx(180.39e9, rel=1e-4)
    assert workloads.D26.fwd_bwd_flops() == pytest.approx(781.68e9, rel=1e-5)


def test_kv_heads_generators_keep_the_multi_head_draws():
    """kv_heads = H (or unset) draws exactly the multi-head tensors, so every
    seeded case keeps its inputs; fewer key/value heads shape k, v (and the
    caches) with that many heads."""
    import torch
    a = workloads.attn_inputs(1, 5, 4, 64, 7)
    b = workloads.attn_inputs(1, 5, 4, 64, 7, kv_heads=4)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    q, k, v, dout = workloads.attn_inputs(1, 5, 4, 64, 7, kv_heads=2)
    assert q.shape == (1, 5, 4, 64) and k.shape == v.shape == (1, 5, 2, 64) and dout.shape == q.shape
    lens, qd, kc, vc = workloads.decode_inputs(2, 6, 64, 16, 8, lens=[3, 16], kv_heads=3)
    assert qd.shape == (2, 6, 64) and kc.shape == vc.shape == (2, 16, 3, 64)
    start, qp, kp, vp = workloads.prefill_inputs(2, 4, 6, 64, 16, 9, start=[0, 12], kv_heads=1)
    assert qp.shape == (2, 4, 6, 64) and kp.shape == vp.shape == (2, 16, 1, 64)
    # algorithmic decode bytes: key and value rows of Hkv heads, q and out of H
    assert workloads.decode_bytes([3, 16], 6, 64, 3) == 19 * 3 * 64 * 4 + 2 * 2 * 6 * 64 * 2 + 8
    assert workloads.decode_bytes([3, 16], 6, 64) == workloads.decode_bytes([3, 16], 6, 64, 6)
