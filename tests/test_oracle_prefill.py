"""Pins for the oracle's chunked prefill (C new tokens per stream at a cache
offset): it must be rows start .. start+C-1 of the forward over the whole
sequence, and each row the single-token decode of that position.  Generation
runs prompts through a KV cache with prefill and decode (ai.flicky.cc,
"nanochat: свой ChatGPT от токенизатора до чата", section "Карта
репозитория", engine.py row)."""
import numpy as np
import pytest

import oracle
from workloads import prefill_inputs


@pytest.mark.parametrize("W", [0, 5])
def test_prefill_from_zero_is_the_forward(W):
    B, C, H, D = 2, 23, 2, 16
    start, q, k_raw, v = prefill_inputs(B, C, H, D, Tcap=C, seed=80, start=[0, 0])
    out, lse = oracle.attn_prefill(q, k_raw, v, start, window=W)
    qf = q.clone()
    o, l = oracle.attn_fwd(qf, k_raw, v, window=W)
    assert np.allclose(out, o, atol=1e-13)
    assert np.allclose(lse, l, atol=1e-13)


@pytest.mark.parametrize("W", [0, 7])
def test_prefill_rows_are_forward_rows_of_the_whole_sequence(W):
    """Queries before the chunk do not influence its rows (causality), so the
    forward over the whole sequence, with the chunk's queries in their rows,
    gives the chunk's outputs in rows start .. start+C-1."""
    B, C, H, D, Tcap = 3, 9, 2, 16, 40
    start, q, k_raw, v = prefill_inputs(B, C, H, D, Tcap, seed=81, start=[0, 13, 31])
    out, lse = oracle.attn_prefill(q, k_raw, v, start, window=W)
    for b, s in enumerate(start.tolist()):
        L = s + C
        qf = k_raw[b:b + 1, :L].clone()  # rows before the chunk are irrelevant
        qf[0, s:L] = q[b]
        o, l = oracle.attn_fwd(qf, k_raw[b:b + 1, :L], v[b:b + 1, :L], window=W)
        assert np.allclose(out[b], o[0, s:L], atol=1e-13)
        assert np.allclose(lse[b], l[0][:, s:L], atol=1e-13)


def test_prefill_row_is_the_decode_of_its_position():
    B, C, H, D, Tcap = 2, 6, 3, 32, 30
    start, q, k_raw, v = prefill_inputs(B, C, H, D, Tcap, seed=82, start=[4, 20])
    out, _ = oracle.attn_prefill(q, k_raw, v, start)
    for t in range(C):
        lens = start + t + 1
        dec = oracle.attn_decode(q[:, t], k_raw, v, lens)
        assert np.allclose(out[:, t], dec, atol=1e-13)


def test_two_chunks_equal_one():
    """Prefilling a sequence in two chunks gives the rows of one forward."""
    B, H, D, T, a = 1, 2, 16, 25, 11
    _, q, k_raw, v = prefill_inputs(B, T, H, D, T, seed=83, start=[0])
    o, _ = oracle.attn_fwd(q, k_raw, v)
    o1, _ = oracle.attn_prefill(q[:, :a], k_raw, v, [0])
    o2, _ = oracle.attn_prefill(q[:, a:], k_raw, v, [a])
    assert np.allclose(np.concatenate([o1, o2], axis=1), o, atol=1e-13)
