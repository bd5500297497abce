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
